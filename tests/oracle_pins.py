"""Pins of the CPU oracle against facts the pages and the mathematics fix.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with:
a worked example derived by hand, a closed form, a special case that reduces to a
plain library routine, an invariant, or brute force written with explicit loops.
They are collected by ``test_oracle_pins.py`` and re-run under planted mistakes by
``test_oracle_mutations.py`` (every planted mistake must trip at least one pin).
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np

from oracle import dspark_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_example.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _f32(x):
    return np.asarray(x, np.float32)


def _hand_inputs(g):
    return dict(hidden=_f32(g["hidden"]), lm_head=_f32(g["lm_head"]),
                markov_w1=_f32(g["markov_w1"]), markov_w2=_f32(g["markov_w2"]),
                w_conf=_f32(g["w_conf"]), b_conf=g["b_conf"])


# --------------------------------------------------------------------------- golden
def pin_hand_anchor_first():
    g = _golden()
    x = _hand_inputs(g)
    e = g["expected"]["anchor_first"]
    o = O.propose(x["hidden"], [g["anchor"]], x["lm_head"], x["markov_w1"],
                  x["markov_w2"], L_in=g["L_in"], sample_from_anchor=True, top_k=2,
                  conf_min=e["conf_min"], w_conf=x["w_conf"], b_conf=x["b_conf"],
                  return_logits=True)
    assert o["draft"][0].tolist() == e["draft"], o["draft"]
    assert np.array_equal(o["logits"][0], np.asarray(e["corrected_logits"], float))
    assert np.allclose(o["conf"][0], e["conf"], rtol=0, atol=1e-15)
    assert int(o["n_draft"][0]) == e["n_draft"]
    assert o["topk_ids"][0].tolist() == e["top2_ids_markov"]
    assert o["topk_vals"][0].tolist() == e["top2_vals_markov"]


def pin_hand_topk_base():
    g = _golden()
    x = _hand_inputs(g)
    e = g["expected"]["anchor_first"]
    o = O.propose(x["hidden"], [g["anchor"]], x["lm_head"], x["markov_w1"],
                  x["markov_w2"], L_in=g["L_in"], sample_from_anchor=True, top_k=2,
                  conf_min=0.0, topk_markov=False)
    assert o["topk_ids"][0].tolist() == e["top2_ids_base"]
    assert o["topk_vals"][0].tolist() == e["top2_vals_base"]
    assert o["draft"][0].tolist() == e["draft"]          # the chain itself is unchanged


def pin_hand_plain_argmax():
    g = _golden()
    x = _hand_inputs(g)
    zero1 = np.zeros_like(x["markov_w1"])
    o = O.propose(x["hidden"], [g["anchor"]], x["lm_head"], zero1, x["markov_w2"],
                  L_in=g["L_in"], sample_from_anchor=True, top_k=1, conf_min=0.0)
    assert o["draft"][0].tolist() == g["expected"]["anchor_first"]["plain_argmax"]


def pin_hand_bonus_anchor():
    g = _golden()
    x = _hand_inputs(g)
    e = g["expected"]["bonus_anchor"]
    o = O.propose(x["hidden"], [g["anchor"]], x["lm_head"], x["markov_w1"],
                  x["markov_w2"], L_in=g["L_in"], sample_from_anchor=False, top_k=1,
                  conf_min=e["conf_min"], w_conf=x["w_conf"], b_conf=x["b_conf"])
    assert o["N"] == g["L_in"] - 1
    assert o["draft"][0].tolist() == e["draft"], o["draft"]
    assert int(o["n_draft"][0]) == e["n_draft"]


def pin_hand_masked_row():
    g = _golden()
    x = _hand_inputs(g)
    e = g["expected"]["masked_row_2"]
    o = O.propose(x["hidden"], [g["anchor"]], x["lm_head"], x["markov_w1"],
                  x["markov_w2"], L_in=g["L_in"], sample_from_anchor=True, top_k=1,
                  conf_min=0.0, lm_bias=_f32(e["lm_bias"]))
    assert o["draft"][0].tolist() == e["draft"], o["draft"]


def pin_hand_verify():
    g = _golden()
    for case in g["expected"]["verify"]:
        a, b, em = O.verify([case["draft"]], [case["n_draft"]], [case["target"]])
        assert int(a[0]) == case["accepted"], (case, a)
        assert int(b[0]) == case["bonus"], (case, b)
        assert em[0].tolist() == case["emitted"], (case, em)


# ------------------------------------------------------------------- brute force
def _brute_force_propose(hidden, anchors, W, w1, w2, bias, L_in, sfa, k, topk_markov=True):
    """The proposal written with explicit loops and a materialised V x V bigram table.
    With topk_markov False the top-k ranks the base logits instead of the corrected ones."""
    h = O.upcast(hidden)
    W = O.upcast(W)
    w1 = O.upcast(w1)
    w2 = O.upcast(w2)
    B, _, H = h.shape
    V, r = w1.shape
    ifp = 0 if sfa else 1
    N = L_in - ifp
    T = [[sum(w1[p][q] * w2[q][v] for q in range(r)) for v in range(V)] for p in range(V)]
    draft = [[0] * N for _ in range(B)]
    topk = [[None] * N for _ in range(B)]
    for b in range(B):
        prev = int(anchors[b])
        for i in range(N):
            row, base = [], []
            for v in range(V):
                s = 0.0
                for c in range(H):
                    s += h[b][ifp + i][c] * W[v][c]
                if bias is not None:
                    s += float(bias[v])
                base.append(s)
                row.append(s + T[prev][v])
            best = 0
            for v in range(1, V):
                if row[v] > row[best]:
                    best = v
            ranked = row if topk_markov else base
            order = sorted(range(V), key=lambda v: (-ranked[v], v))[:k]
            draft[b][i] = best
            topk[b][i] = (order, [ranked[v] for v in order])
            prev = best
    return draft, topk


def pin_brute_force_tiny(dtype="bf16", sfa=True, with_bias=False):
    from workloads import Workload, make_head, make_batch
    wl = Workload("bf", B=3, L_in=3, H=8, V=64, r=4, top_k=3, sample_from_anchor=sfa,
                  conf_min=0.0, dtype=dtype, weight_std=0.5, conf_std=0.5,
                  n_emit=40 if with_bias else None, seed=77)
    hd = make_head(wl)
    bt = make_batch(wl)
    o = O.propose(bt["hidden"], bt["anchors"], hd["lm_head"], hd["markov_w1"],
                  hd["markov_w2"], L_in=wl.L_in, sample_from_anchor=sfa, top_k=3,
                  conf_min=0.0, lm_bias=hd["lm_bias"])
    d, tk = _brute_force_propose(bt["hidden"], bt["anchors"], hd["lm_head"],
                                 hd["markov_w1"], hd["markov_w2"], hd["lm_bias"],
                                 wl.L_in, sfa, 3)
    assert o["draft"].tolist() == d, (o["draft"], d)
    for b in range(wl.B):
        for i in range(wl.N):
            assert o["topk_ids"][b, i].tolist() == tk[b][i][0]
            assert np.allclose(o["topk_vals"][b, i], tk[b][i][1], rtol=1e-12, atol=1e-9)


def pin_brute_force_variants():
    pin_brute_force_tiny("f32", True, False)
    pin_brute_force_tiny("bf16", False, False)
    pin_brute_force_tiny("bf16", True, True)


def pin_adaptive_block_length():
    """skip_truncated: slots before the confidence cut are the brute-force proposal's,
    slots from the cut on read -1 (top-k values NaN), and verify cannot tell the two
    apart, since it reads nothing past the cut."""
    from workloads import Workload, make_head, make_batch
    wl = Workload("ad", B=4, L_in=5, H=8, V=64, r=4, top_k=3, sample_from_anchor=True,
                  conf_min=0.5, dtype="f32", weight_std=0.5, conf_std=0.5, seed=78)
    hd = make_head(wl)
    bt = make_batch(wl)
    # hidden column 0 and a one-hot w_conf put block b's cut at slot cuts[b]
    cuts = [0, 2, 4, 5]
    hidden = np.array(bt["hidden"], np.float32)
    w_conf = np.zeros(wl.H, np.float32)
    w_conf[0] = 1.0
    for b, c in enumerate(cuts):
        hidden[b, :, 0] = 2.0
        if c < wl.L_in:
            hidden[b, c, 0] = -2.0
    kw = dict(L_in=wl.L_in, sample_from_anchor=True, top_k=3, conf_min=0.5, w_conf=w_conf)
    o = O.propose(hidden, bt["anchors"], hd["lm_head"], hd["markov_w1"], hd["markov_w2"],
                  skip_truncated=True, **kw)
    full = O.propose(hidden, bt["anchors"], hd["lm_head"], hd["markov_w1"],
                     hd["markov_w2"], **kw)
    d, tk = _brute_force_propose(hidden, bt["anchors"], hd["lm_head"], hd["markov_w1"],
                                 hd["markov_w2"], None, wl.L_in, True, 3)
    assert o["n_draft"].tolist() == cuts
    for b, c in enumerate(cuts):
        assert o["draft"][b, :c].tolist() == d[b][:c]
        assert (o["draft"][b, c:] == -1).all()
        assert (o["topk_ids"][b, c:] == -1).all() and np.isnan(o["topk_vals"][b, c:]).all()
        for i in range(c):
            assert o["topk_ids"][b, i].tolist() == tk[b][i][0]
    rng = np.random.default_rng(5)
    for _ in range(20):
        target = rng.integers(0, wl.V, (wl.B, wl.N + 1))
        target[:, :2] = np.where(rng.uniform(size=(wl.B, 2)) < 0.7,
                                 np.maximum(full["draft"][:, :2], 0), target[:, :2])
        a1, b1, e1 = O.verify(o["draft"], o["n_draft"], target)
        a2, b2, e2 = O.verify(full["draft"], full["n_draft"], target)
        assert a1.tolist() == a2.tolist() and b1.tolist() == b2.tolist()
        assert np.array_equal(e1, e2)


# ------------------------------------------------------------ special cases / forms
def pin_zero_markov_is_plain_argmax():
    """w1 = w2 = 0 reduces DSpark to the plain lm_head argmax (DFlash's projection)."""
    rng = np.random.default_rng(5)
    B, L, H, V, r = 4, 5, 16, 300, 8
    hidden = rng.standard_normal((B, L, H)).astype(np.float32)
    W = rng.standard_normal((V, H)).astype(np.float32)
    bias = rng.standard_normal(V).astype(np.float32)
    zeros1 = np.zeros((V, r), np.float32)
    zeros2 = np.zeros((r, V), np.float32)
    anchors = rng.integers(0, V, B)
    o = O.propose(hidden, anchors, W, zeros1, zeros2, L_in=L, sample_from_anchor=True,
                  top_k=1, conf_min=0.0, lm_bias=bias)
    plain = np.argmax(hidden.astype(np.float64) @ W.astype(np.float64).T + bias, axis=-1)
    assert np.array_equal(o["draft"], plain)


def pin_one_hot_markov_row():
    """w1[p] = e_j makes the Markov term of prev = p exactly row j of markov_w2."""
    rng = np.random.default_rng(6)
    V, r = 50, 6
    w1 = np.zeros((V, r), np.float32)
    w1[17, 4] = 1.0
    w2 = rng.standard_normal((r, V)).astype(np.float32)
    mk = O.markov_bias(w1, O.upcast(w2), 17)
    assert np.array_equal(mk, w2[4].astype(np.float64))
    w1[17, 4] = -2.0
    assert np.array_equal(O.markov_bias(w1, O.upcast(w2), 17), -2.0 * w2[4].astype(np.float64))


def pin_chain_consistency():
    """Each slot's token is the corrected argmax given the previous slot's token."""
    rng = np.random.default_rng(7)
    B, L, H, V, r = 3, 6, 12, 97, 5
    hidden = rng.standard_normal((B, L, H)).astype(np.float32)
    W = rng.standard_normal((V, H)).astype(np.float32)
    w1 = rng.standard_normal((V, r)).astype(np.float32) * 2
    w2 = rng.standard_normal((r, V)).astype(np.float32) * 2
    anchors = rng.integers(0, V, B)
    o = O.propose(hidden, anchors, W, w1, w2, L_in=L, sample_from_anchor=True,
                  top_k=1, conf_min=0.0, return_logits=True)
    h = hidden.astype(np.float64)
    for b in range(B):
        prev = anchors[b]
        for i in range(L):
            row = h[b, i] @ W.astype(np.float64).T
            row = row + w1[prev].astype(np.float64) @ w2.astype(np.float64)
            assert int(np.argmax(row)) == o["draft"][b, i]
            prev = o["draft"][b, i]
    # the Markov term matters in this case (otherwise this pin would be vacuous)
    o0 = O.propose(hidden, anchors, W, np.zeros_like(w1), w2, L_in=L,
                   sample_from_anchor=True, top_k=1, conf_min=0.0)
    assert not np.array_equal(o0["draft"], o["draft"])


def pin_single_slot():
    """L = 1: one corrected argmax whose previous token is the anchor."""
    rng = np.random.default_rng(8)
    H, V, r = 10, 40, 3
    hidden = rng.standard_normal((2, 1, H)).astype(np.float32)
    W = rng.standard_normal((V, H)).astype(np.float32)
    w1 = rng.standard_normal((V, r)).astype(np.float32) * 3
    w2 = rng.standard_normal((r, V)).astype(np.float32) * 3
    anchors = np.array([3, 39])
    o = O.propose(hidden, anchors, W, w1, w2, L_in=1, sample_from_anchor=True,
                  top_k=1, conf_min=0.0)
    for b in range(2):
        row = hidden[b, 0].astype(np.float64) @ W.T.astype(np.float64) \
            + w1[anchors[b]].astype(np.float64) @ w2.astype(np.float64)
        assert o["draft"][b, 0] == int(np.argmax(row))


def pin_masked_rows_never_emitted():
    """Rows biased by -1e9 never become a draft token or a top-k candidate (k <= V_e)."""
    rng = np.random.default_rng(9)
    B, L, H, V, r, Ve, k = 4, 4, 16, 500, 8, 37, 5
    hidden = rng.standard_normal((B, L, H)).astype(np.float32)
    W = rng.standard_normal((V, H)).astype(np.float32) * 3
    w1 = rng.standard_normal((V, r)).astype(np.float32)
    w2 = rng.standard_normal((r, V)).astype(np.float32)
    emit = np.sort(rng.choice(V, Ve, replace=False))
    bias = np.full(V, -1e9, np.float32)
    bias[emit] = 0
    o = O.propose(hidden, rng.integers(0, V, B), W, w1, w2, L_in=L, sample_from_anchor=False,
                  top_k=k, conf_min=0.0, lm_bias=bias)
    ok = set(emit.tolist())
    assert set(o["draft"].ravel().tolist()) <= ok
    assert set(o["topk_ids"].ravel().tolist()) <= ok


def pin_confidence_closed_forms():
    rng = np.random.default_rng(10)
    hidden = rng.standard_normal((2, 3, 8)).astype(np.float32)
    zero = np.zeros(8, np.float32)
    assert np.all(O.confidence(hidden, zero, 0.0, 0, 3) == 0.5)
    assert np.allclose(O.confidence(hidden, zero, 40.0, 0, 3), 1.0, rtol=0, atol=1e-15)
    assert np.allclose(O.confidence(hidden, zero, -40.0, 0, 3), 4.248354255291589e-18,
                       rtol=1e-12, atol=0)
    assert np.allclose(O.confidence(hidden, zero, 1.0, 0, 3), 1 / (1 + math.exp(-1)),
                       rtol=1e-15, atol=0)
    # a one-hot w_conf reads one hidden coordinate of the slot (offset by the layout)
    e = np.zeros(8, np.float32)
    e[2] = 1.0
    c = O.confidence(hidden, e, 0.0, 1, 2)
    want = 1 / (1 + np.exp(-hidden[:, 1:3, 2].astype(np.float64)))
    assert np.allclose(c, want, rtol=1e-15, atol=0)


def pin_truncation_positions():
    """The first slot below the threshold cuts the block; equality keeps the slot."""
    N = 6
    rng = np.random.default_rng(13)
    for j in range(N + 1):
        conf = np.full(N, 0.9)
        if j < N:
            conf[j] = 0.1
            conf[j + 1:] = rng.uniform(0, 1, N - j - 1)   # whatever follows the cut
        assert O.truncation_length(conf, 0.5) == j
    conf = np.array([0.5, 0.5, 0.49, 0.9])
    assert O.truncation_length(conf, 0.5) == 2
    assert O.truncation_length(np.array([0.0, 0.0]), 0.0) == 2   # 0 disables
    assert O.truncation_length(np.array([0.2, 0.9]), -1.0) == 2
    # crafted through the confidence head: slot j's logit is set via a one-hot w_conf
    B, L, H = 1, 6, 4
    for j in range(L):
        hidden = np.zeros((B, L, H), np.float32)
        hidden[0, :, 0] = 1.0
        hidden[0, j, 0] = -1.0
        c = O.confidence(hidden, np.array([1, 0, 0, 0], np.float32), 0.0, 0, L)
        assert O.truncation_length(c[0], 0.5) == j


def pin_verify_brute_force():
    """All drafts/targets over V=3, N=3 and every n_draft: accept = common prefix."""
    V, N = 3, 3
    for d in itertools.product(range(V), repeat=N):
        for t in itertools.product(range(V), repeat=N + 1):
            for nd in range(N + 1):
                a, bo, em = O.verify([d], [nd], [t])
                # independent form: count leading matches among the first nd slots
                eq = [d[j] == t[j] for j in range(nd)] + [False]
                want = eq.index(False)
                assert int(a[0]) == want
                assert int(bo[0]) == t[want]
                # greedy lossless: what is emitted is the target's own argmax sequence
                assert em[0, :want + 1].tolist() == list(t[:want + 1])
                assert all(x == -1 for x in em[0, want + 1:])


def pin_verify_planted_mismatch():
    rng = np.random.default_rng(11)
    N, V = 16, 1000
    for nd in (0, 5, 16):
        for j in range(N):
            d = rng.integers(0, V, N)
            t = np.concatenate([d, rng.integers(0, V, 1)])
            t[j] = (d[j] + 1) % V
            a, bo, _ = O.verify([d], [nd], [t])
            assert int(a[0]) == min(j, nd)
            assert int(bo[0]) == t[min(j, nd)]


def pin_bf16_upcast():
    bits = np.array([0x3F80, 0xC000, 0x3E80, 0x0000, 0x8000, 0x4049, 0x7F7F], np.uint16)
    want = [1.0, -2.0, 0.25, 0.0, -0.0, 3.140625, 3.3895313892515355e38]
    got = O.upcast(bits)
    assert got.tolist() == want, got


def pin_bonus_slot_unused():
    """In the 1+N layout the bonus slot's hidden state influences nothing."""
    rng = np.random.default_rng(12)
    B, L, H, V, r = 2, 5, 8, 60, 4
    hidden = rng.standard_normal((B, L, H)).astype(np.float32)
    W = rng.standard_normal((V, H)).astype(np.float32)
    w1 = rng.standard_normal((V, r)).astype(np.float32)
    w2 = rng.standard_normal((r, V)).astype(np.float32)
    wc = rng.standard_normal(H).astype(np.float32)
    anchors = rng.integers(0, V, B)
    kw = dict(L_in=L, sample_from_anchor=False, top_k=2, conf_min=0.5, w_conf=wc)
    o1 = O.propose(hidden, anchors, W, w1, w2, **kw)
    h2 = hidden.copy()
    h2[:, 0, :] = rng.standard_normal((B, H)) * 10
    o2 = O.propose(h2, anchors, W, w1, w2, **kw)
    assert o1["N"] == L - 1
    for key in ("draft", "topk_ids", "n_draft"):
        assert np.array_equal(o1[key], o2[key])
    # ... whereas changing the first prediction slot's hidden state does matter
    h3 = hidden.copy()
    h3[:, 1, :] = -h3[:, 1, :] * 5
    o3 = O.propose(h3, anchors, W, w1, w2, **kw)
    assert not np.array_equal(o1["draft"][:, 0], o3["draft"][:, 0])


# ------------------------------------------------------------------- tree verify
def _random_lattice(rng, B, N, k, V):
    """Top-k ids of distinct tokens per slot, as the proposal produces them."""
    return np.array([[rng.choice(V, k, replace=False) for _ in range(N)]
                     for _ in range(B)], np.int64)


def _tree_brute_force(ids_b, nd, t):
    """Every node of the candidate tree, written out: a node is the tuple of candidate
    ranks taken at depths 0..d-1 (d <= nd).  The greedy target reaches a node when the
    node's tokens equal its own tokens t[0..d-1]; it accepts the deepest such node."""
    N, k = ids_b.shape
    best, best_ranks = 0, ()
    for d in range(nd + 1):
        for ranks in itertools.product(range(k), repeat=d):
            tokens = [int(ids_b[i, ranks[i]]) for i in range(d)]
            if tokens == [int(x) for x in t[:d]] and d >= best:
                best, best_ranks = d, ranks
    return best, best_ranks


def pin_tree_verify_brute_force():
    rng = np.random.default_rng(21)
    V, N = 4, 3
    for k in (1, 2, 3):
        for _ in range(3):
            ids = _random_lattice(rng, 1, N, k, V)
            for t in itertools.product(range(V), repeat=N + 1):
                for nd in range(N + 1):
                    a, bo, em, path = O.tree_verify(ids, [nd], [t])
                    want, ranks = _tree_brute_force(ids[0], nd, t)
                    assert int(a[0]) == want, (ids, t, nd)
                    assert int(bo[0]) == t[want]
                    # greedy lossless: the target's own tokens, then -1
                    assert em[0, :want + 1].tolist() == list(t[:want + 1])
                    assert all(x == -1 for x in em[0, want + 1:])
                    assert path[0, :want].tolist() == list(ranks)
                    assert all(x == -1 for x in path[0, want:])


def pin_tree_verify_top1_is_verify():
    """With one candidate per slot the lattice is the greedy draft itself."""
    rng = np.random.default_rng(22)
    B, N, V = 5, 6, 5
    for _ in range(50):
        ids = rng.integers(0, V, (B, N, 1))
        t = rng.integers(0, V, (B, N + 1))
        t[:, :3] = np.where(rng.random((B, 3)) < 0.6, ids[:, :3, 0], t[:, :3])
        nd = rng.integers(0, N + 1, B)
        a, bo, em, _ = O.tree_verify(ids, nd, t)
        a2, bo2, em2 = O.verify(ids[:, :, 0], nd, t)
        assert np.array_equal(a, a2) and np.array_equal(bo, bo2) and np.array_equal(em, em2)


def pin_tree_verify_planted_miss():
    """The target's token at depth j is in no candidate of that depth: accepted
    min(j, n_draft), whichever ranks matched before it."""
    rng = np.random.default_rng(23)
    N, k, V = 8, 4, 100
    for nd in (0, 3, 8):
        for j in range(N):
            ids = _random_lattice(rng, 1, N, k, V)
            ranks = rng.integers(0, k, N)
            t = np.array([ids[0, i, ranks[i]] for i in range(N)] + [7])
            t[j] = next(x for x in range(V) if x not in ids[0, j])
            a, bo, _, path = O.tree_verify(ids, [nd], [t])
            assert int(a[0]) == min(j, nd)
            assert int(bo[0]) == t[min(j, nd)]
            assert path[0, :min(j, nd)].tolist() == ranks[:min(j, nd)].tolist()


# ------------------------------------------------------------------- conf input
def pin_separate_confidence_input():
    """A separate confidence input changes the confidences (closed form with a one-hot
    w_conf) and nothing else; given the hidden states themselves it changes nothing."""
    rng = np.random.default_rng(24)
    B, L, H, V, r = 3, 5, 8, 50, 4
    hidden = rng.standard_normal((B, L, H)).astype(np.float32)
    ch = rng.standard_normal((B, L, H)).astype(np.float32)
    W = rng.standard_normal((V, H)).astype(np.float32)
    w1 = rng.standard_normal((V, r)).astype(np.float32)
    w2 = rng.standard_normal((r, V)).astype(np.float32)
    wc = np.zeros(H, np.float32)
    wc[2] = 1.0
    anchors = rng.integers(0, V, B)
    for sfa in (True, False):
        kw = dict(L_in=L, sample_from_anchor=sfa, top_k=3, conf_min=0.5, w_conf=wc,
                  b_conf=0.25)
        base = O.propose(hidden, anchors, W, w1, w2, **kw)
        same = O.propose(hidden, anchors, W, w1, w2, conf_hidden=hidden, **kw)
        other = O.propose(hidden, anchors, W, w1, w2, conf_hidden=ch, **kw)
        for key in ("draft", "topk_ids", "topk_vals", "conf", "n_draft"):
            assert np.array_equal(base[key], same[key]), key
        for key in ("draft", "topk_ids", "topk_vals"):
            assert np.array_equal(base[key], other[key]), key
        ifp = 0 if sfa else 1
        N = base["N"]
        want = 1.0 / (1.0 + np.exp(-(ch[:, ifp:ifp + N, 2].astype(np.float64) + 0.25)))
        assert np.allclose(other["conf"], want, rtol=0, atol=1e-15)
        cut = [next((i for i in range(N) if want[b, i] < 0.5), N) for b in range(B)]
        assert other["n_draft"].tolist() == cut


# ------------------------------------------------------------------- random sweep
def sweep_case(seed):
    """A random tiny configuration with small-integer weights and hidden states: every
    logit is exact in float64 and exact ties are common, so the tie rules get exercised.
    Covers both layouts, both top-k sources, masked rows and the confidence threshold
    (sometimes exactly equal to a slot's confidence)."""
    rng = np.random.default_rng(10_000 + seed)
    sfa = bool(rng.integers(0, 2))
    B = int(rng.integers(1, 3))
    L_in = int(rng.integers(1 if sfa else 2, 5))
    H = int(rng.integers(1, 4))
    V = int(rng.integers(2, 10))
    r = int(rng.integers(1, 4))

    def ints(*shape):
        return rng.integers(-2, 3, size=shape).astype(np.float32)

    hidden, W = ints(B, L_in, H), ints(V, H)
    w1, w2 = ints(V, r), ints(r, V)
    bias = None
    if rng.integers(0, 2):
        bias = np.zeros(V, np.float32)
        masked = rng.choice(V, size=int(rng.integers(0, V // 2 + 1)), replace=False)
        bias[masked] = np.float32(-1e9)
    n_emit = V if bias is None else int(np.sum(bias > -1e8))
    k = int(rng.integers(1, n_emit + 1))
    anchors = rng.integers(0, V, size=B)
    w_conf = ints(H)
    b_conf = float(rng.integers(-1, 2))
    conf_min = [0.0, 0.5, 1.0 / (1.0 + math.exp(-1.0)), 0.9][int(rng.integers(0, 4))]
    topk_markov = bool(rng.integers(0, 2))
    return dict(sfa=sfa, B=B, L_in=L_in, V=V, hidden=hidden, W=W, w1=w1, w2=w2, bias=bias,
                k=k, anchors=anchors, w_conf=w_conf, b_conf=b_conf, conf_min=conf_min,
                topk_markov=topk_markov)


def brute_force_confidence(hidden, w_conf, b_conf, ifp, N, conf_min):
    """Per-slot sigmoid confidence and the first slot strictly below conf_min, in loops."""
    B, _, H = hidden.shape
    conf = [[0.0] * N for _ in range(B)]
    n_draft = []
    for b in range(B):
        for i in range(N):
            x = sum(float(hidden[b, ifp + i, c]) * float(w_conf[c]) for c in range(H))
            conf[b][i] = 1.0 / (1.0 + math.exp(-(x + b_conf)))
        cut = N
        if conf_min > 0:
            for i in range(N):
                if conf[b][i] < conf_min:
                    cut = i
                    break
        n_draft.append(cut)
    return conf, n_draft


def check_sweep_case(seed):
    c = sweep_case(seed)
    o = O.propose(c["hidden"], c["anchors"], c["W"], c["w1"], c["w2"], L_in=c["L_in"],
                  sample_from_anchor=c["sfa"], top_k=c["k"], conf_min=c["conf_min"],
                  lm_bias=c["bias"], w_conf=c["w_conf"], b_conf=c["b_conf"],
                  topk_markov=c["topk_markov"])
    d, tk = _brute_force_propose(c["hidden"], c["anchors"], c["W"], c["w1"], c["w2"],
                                 c["bias"], c["L_in"], c["sfa"], c["k"], c["topk_markov"])
    ifp = 0 if c["sfa"] else 1
    N = c["L_in"] - ifp
    assert o["draft"].tolist() == d, (seed, o["draft"], d)
    for b in range(c["B"]):
        for i in range(N):
            assert o["topk_ids"][b, i].tolist() == tk[b][i][0], (seed, b, i)
            assert o["topk_vals"][b, i].tolist() == tk[b][i][1], (seed, b, i)
            if c["bias"] is not None:
                assert c["bias"][o["draft"][b, i]] > -1e8, (seed, b, i)
    conf, n_draft = brute_force_confidence(c["hidden"], c["w_conf"], c["b_conf"], ifp, N,
                                           c["conf_min"])
    assert np.allclose(o["conf"], conf, rtol=0, atol=1e-15), seed
    assert o["n_draft"].tolist() == n_draft, (seed, o["n_draft"], n_draft)


def pin_brute_force_sweep():
    for seed in range(40):
        check_sweep_case(seed)


ALL_PINS = [
    pin_hand_anchor_first, pin_hand_topk_base, pin_hand_plain_argmax,
    pin_hand_bonus_anchor, pin_hand_masked_row, pin_hand_verify,
    pin_brute_force_variants, pin_zero_markov_is_plain_argmax, pin_one_hot_markov_row,
    pin_chain_consistency, pin_single_slot, pin_masked_rows_never_emitted,
    pin_confidence_closed_forms, pin_truncation_positions, pin_verify_brute_force,
    pin_verify_planted_mismatch, pin_bf16_upcast, pin_bonus_slot_unused,
    pin_adaptive_block_length, pin_brute_force_sweep, pin_tree_verify_brute_force,
    pin_tree_verify_top1_is_verify, pin_tree_verify_planted_miss,
    pin_separate_confidence_input,
]
