"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin fails.

A pin set that a dropped term, a flipped sign, a wrong index or a transposed operand
can slip through would not be evidence that the oracle is right.
"""
import contextlib

import numpy as np
import pytest

import oracle_pins
from oracle import dspark_oracle as O


def _argmax_highest(row):
    m = row.max()
    return int(np.flatnonzero(row == m)[-1])


def _chain_prev_always_anchor(z_b, w1, w2_f64, anchor, top_k=1, topk_markov=True):
    N, V = z_b.shape
    tok = np.empty(N, np.int64)
    ids = np.empty((N, top_k), np.int64)
    vals = np.empty((N, top_k))
    zc = np.empty_like(z_b)
    for i in range(N):
        zc[i] = O.corrected_logits(z_b[i], w1, w2_f64, int(anchor))
        tok[i] = O.argmax_lowest(zc[i])
        ranked = zc[i] if topk_markov else z_b[i]
        ids[i] = O.topk_sorted(ranked, top_k)
        vals[i] = ranked[ids[i]]
    return tok, ids, vals, zc


def _chain_prev_is_own_slot(z_b, w1, w2_f64, anchor, top_k=1, topk_markov=True):
    """prev(i) taken from the base argmax of slot i itself (an indexing slip)."""
    N, V = z_b.shape
    tok = np.empty(N, np.int64)
    ids = np.empty((N, top_k), np.int64)
    vals = np.empty((N, top_k))
    zc = np.empty_like(z_b)
    for i in range(N):
        prev = int(anchor) if i == 0 else O.argmax_lowest(z_b[i])
        zc[i] = O.corrected_logits(z_b[i], w1, w2_f64, prev)
        tok[i] = O.argmax_lowest(zc[i])
        ranked = zc[i] if topk_markov else z_b[i]
        ids[i] = O.topk_sorted(ranked, top_k)
        vals[i] = ranked[ids[i]]
    return tok, ids, vals, zc


def _verify_no_ndraft(draft, n_draft, target):
    return _orig_verify(draft, np.full(len(draft), np.asarray(draft).shape[1]), target)


def _verify_bonus_next(draft, n_draft, target):
    a, b, e = _orig_verify(draft, n_draft, target)
    t = np.asarray(target)
    b2 = np.array([t[i, min(a[i] + 1, t.shape[1] - 1)] for i in range(len(a))])
    e = e.copy()
    for i in range(len(a)):
        e[i, a[i]] = b2[i]
    return a, b2, e


_orig_verify = O.verify
_orig_layout = O.block_layout
_orig_base = O.base_logits
_orig_conf = O.confidence
_orig_blank = O.blank_past_cut


MUTATIONS = {
    "markov_dropped": ("corrected_logits", lambda z, w1, w2, prev: z),
    "markov_sign": ("corrected_logits",
                    lambda z, w1, w2, prev: z - O.markov_bias(w1, w2, prev)),
    "markov_columns_reversed": ("markov_bias",
                                lambda w1, w2, prev: O.upcast(np.asarray(w1)[prev]) @ w2[:, ::-1]),
    "markov_rank_dropped": ("markov_bias",
                            lambda w1, w2, prev: O.upcast(np.asarray(w1)[prev])[..., :-1] @ w2[:-1]),
    "tie_to_highest": ("argmax_lowest", _argmax_highest),
    "topk_ascending": ("topk_sorted",
                       lambda row, k: np.lexsort((np.arange(row.shape[-1]), row))[:k]),
    "prev_always_anchor": ("greedy_chain", _chain_prev_always_anchor),
    "prev_from_own_slot": ("greedy_chain", _chain_prev_is_own_slot),
    "truncate_le": ("truncation_length",
                    lambda c, m: next((i for i in range(len(c)) if m > 0 and c[i] <= m), len(c))),
    "conf_bias_dropped": ("confidence",
                          lambda h, w, b, ifp, N: _orig_conf(h, w, 0.0, ifp, N)),
    "conf_sign": ("confidence",
                  lambda h, w, b, ifp, N: 1 - _orig_conf(h, w, b, ifp, N)),
    "layout_bonus_ignored": ("block_layout", lambda L, sfa: (L, 0)),
    "layout_wrong_offset": ("block_layout", lambda L, sfa: (L, 0) if sfa else (L - 1, 0)),
    "lm_bias_dropped": ("base_logits",
                        lambda h, W, bias, ifp, N, chunk=16384: _orig_base(h, W, None, ifp, N, chunk)),
    "lm_head_transposed_rows": ("base_logits",
                                lambda h, W, bias, ifp, N, chunk=16384:
                                _orig_base(h, np.asarray(W)[:, ::-1], bias, ifp, N, chunk)),
    "verify_ignores_ndraft": ("verify", _verify_no_ndraft),
    "adaptive_cut_one_late": ("blank_past_cut",
                              lambda d, i, v, nd: _orig_blank(d, i, v, np.asarray(nd) + 1)),
    "adaptive_cut_one_early": ("blank_past_cut",
                               lambda d, i, v, nd: _orig_blank(d, i, v, np.maximum(np.asarray(nd) - 1, 0))),
    "verify_bonus_off_by_one": ("verify", _verify_bonus_next),
    "upcast_truncates": ("upcast",
                         lambda a: (np.asarray(a).astype(np.float32).astype(np.float16).astype(np.float64)
                                    if np.asarray(a).dtype != np.uint16 else
                                    ((np.asarray(a).astype(np.uint32) << 16).view(np.float32) * 1.0078125).astype(np.float64))),
}


def _chain_variant(ranked_from=None, vals_from=None, markov_at=None, prev_lag=0):
    """greedy_chain with one planted slip: top-k ranked on the wrong logits, top-k values
    read from the other logits than their ids, the Markov term only at some slots, or the
    previous token taken `prev_lag` slots too early."""
    def chain(z_b, w1, w2_f64, anchor, top_k=1, topk_markov=True):
        N, V = z_b.shape
        tok = np.empty(N, np.int64)
        ids = np.empty((N, top_k), np.int64)
        vals = np.empty((N, top_k))
        zc = np.empty_like(z_b)
        history = [int(anchor)]
        for i in range(N):
            prev = history[max(0, len(history) - 1 - prev_lag)]
            if markov_at is None or markov_at(i):
                zc[i] = O.corrected_logits(z_b[i], w1, w2_f64, prev)
            else:
                zc[i] = z_b[i]
            tok[i] = O.argmax_lowest(zc[i])
            use_markov = topk_markov if ranked_from is None else ranked_from(topk_markov)
            ranked = zc[i] if use_markov else z_b[i]
            ids[i] = O.topk_sorted(ranked, top_k)
            src = ranked if vals_from is None else (z_b[i] if use_markov else zc[i])
            vals[i] = src[ids[i]]
            history.append(int(tok[i]))
        return tok, ids, vals, zc
    return chain


def _truncate_last_below(c, m):
    below = [i for i in range(len(c)) if m > 0 and c[i] < m]
    return below[-1] if below else len(c)


def _verify_counts_matches(draft, n_draft, target):
    d, t = np.asarray(draft), np.asarray(target)
    B, N = d.shape
    a = np.array([int(np.sum(d[b, :n_draft[b]] == t[b, :n_draft[b]])) for b in range(B)])
    bonus = np.array([t[b, a[b]] for b in range(B)])
    e = np.full((B, N + 1), -1, np.int64)
    for b in range(B):
        e[b, :a[b]] = d[b, :a[b]]
        e[b, a[b]] = bonus[b]
    return a, bonus, e


MUTATIONS.update({
    "topk_markov_inverted": ("greedy_chain", _chain_variant(ranked_from=lambda tm: not tm)),
    "topk_markov_always": ("greedy_chain", _chain_variant(ranked_from=lambda tm: True)),
    "topk_vals_from_other_logits": ("greedy_chain", _chain_variant(vals_from=True)),
    "markov_only_first_slot": ("greedy_chain", _chain_variant(markov_at=lambda i: i == 0)),
    "markov_skips_first_slot": ("greedy_chain", _chain_variant(markov_at=lambda i: i > 0)),
    "prev_one_slot_stale": ("greedy_chain", _chain_variant(prev_lag=1)),
    "conf_slot_offset_dropped": ("confidence",
                                 lambda h, w, b, ifp, N: _orig_conf(h, w, b, 0, N)),
    "base_slot_offset_dropped": ("base_logits",
                                 lambda h, W, bias, ifp, N, chunk=8192:
                                 _orig_base(h, W, bias, 0, N, chunk)),
    "truncate_at_last_below": ("truncation_length", _truncate_last_below),
    "verify_counts_matches": ("verify", _verify_counts_matches),
})


_orig_tree = O.tree_verify
_orig_propose = O.propose


def _tree_top1_only(ids, nd, t):
    return _orig_tree(np.asarray(ids)[:, :, :1], nd, t)


def _tree_ignores_ndraft(ids, nd, t):
    return _orig_tree(ids, np.full(len(nd), np.asarray(ids).shape[1]), t)


def _tree_bonus_next(ids, nd, t):
    a, b, e, p = _orig_tree(ids, nd, t)
    t = np.asarray(t)
    b2 = np.array([t[i, min(a[i] + 1, t.shape[1] - 1)] for i in range(len(a))])
    e = e.copy()
    for i in range(len(a)):
        e[i, a[i]] = b2[i]
    return a, b2, e, p


def _tree_next_depth(ids, nd, t):
    """candidates of depth i compared with the target's token of depth i + 1"""
    t = np.asarray(t)
    return _orig_tree(ids, nd, np.concatenate([t[:, 1:], t[:, -1:]], axis=1))


def _tree_rank_reported_last(ids, nd, t):
    a, b, e, p = _orig_tree(ids, nd, t)
    k = np.asarray(ids).shape[2]
    return a, b, e, np.where(p >= 0, k - 1 - p, p)


MUTATIONS.update({
    "tree_top1_only": ("tree_verify", _tree_top1_only),
    "tree_ignores_ndraft": ("tree_verify", _tree_ignores_ndraft),
    "tree_bonus_off_by_one": ("tree_verify", _tree_bonus_next),
    "tree_depth_slip": ("tree_verify", _tree_next_depth),
    "tree_path_rank_flipped": ("tree_verify", _tree_rank_reported_last),
    "conf_hidden_ignored": ("propose",
                            lambda *a, conf_hidden=None, **kw: _orig_propose(*a, **kw)),
    "conf_hidden_feeds_logits": ("propose",
                                 lambda h, *a, conf_hidden=None, **kw:
                                 _orig_propose(h if conf_hidden is None else conf_hidden,
                                               *a, conf_hidden=conf_hidden, **kw)),
})


@contextlib.contextmanager
def _planted(name, fn):
    old = getattr(O, name)
    setattr(O, name, fn)
    try:
        yield
    finally:
        setattr(O, name, old)


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_planted_mistake_is_caught(mutation):
    name, fn = MUTATIONS[mutation]
    caught = []
    with _planted(name, fn), np.errstate(all="ignore"):
        for pin in oracle_pins.ALL_PINS:
            try:
                pin()
            except (AssertionError, IndexError, ValueError):
                caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {mutation}"
