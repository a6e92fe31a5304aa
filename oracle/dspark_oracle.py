"""Plain fp64 CPU oracle of the DSpark proposal head and the greedy verify step.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
benchmark's CPU-baseline leg may import this module; the library's product path
never calls it, and it shares no code with the CUDA path.

Everything is computed in float64 from the exact values the GPU sees (fp32 inputs, or
bf16 bit patterns upcast without rounding).  Each function follows one statement of
the pages; the citation is in its docstring.  The pages used:

  [dflash-log]  llama.cpp commit 6fed9f6 (src/models/dflash.cpp), squash log of
                "spec: add DSpark speculative decoding" and its follow-up commits
  [spec-pr]     llama.cpp PR #26275, "dspark: support speculators-format checkpoints"
  [ort-pr]      onnxruntime-genai PR #2490, "Export DSpark block drafters for Qwen 3.5
                and 3.8", DSpark builder commit message
  [luce-pr]     lucebox PR #626, "feat(qwen38): add adaptive concurrent DSpark
                speculation", description

Readings taken where the pages are silent (each is also listed in the design notes):
  * argmax and top-k ties go to the lowest token id;
  * top-k is ordered by value, descending;
  * the Markov term is the plain rank-r product (no scale, no activation), with
    markov_w1 stored [V, r] (gathered by the previous token) and markov_w2 [r, V];
  * truncation compares strictly (a slot whose confidence equals conf_min is kept);
    conf_min <= 0 disables it; confidence is per slot, not a running product;
  * in the 1+N layout, the first prediction slot's previous token is the anchor;
  * top-k candidates of every slot take the Markov term of the chain's own previous
    token (the greedy path), as the chain's argmax does;
  * the candidate tree that tree verify walks is the whole top-k lattice: every
    candidate of slot i is a child of every candidate of slot i - 1, down to the
    truncated draft length;
  * a separate confidence input (conf_hidden), when given, replaces the hidden states
    in the confidence head only, slot for slot.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "upcast", "block_layout", "base_logits", "markov_bias", "corrected_logits",
    "confidence", "truncation_length", "topk_sorted", "argmax_lowest",
    "greedy_chain", "propose", "verify", "tree_verify", "MASK_BIAS_LIMIT",
]

# A bias at or below this value marks a row the reduced-vocabulary draft cannot emit
# ([spec-pr]: such rows carry -1e9).
MASK_BIAS_LIMIT = -1e8


def upcast(a) -> np.ndarray:
    """Exact float64 copy of an fp32 array or of a bf16 array given as uint16 bits.

    Not a step of the method: bf16 is the upper half of an fp32, so widening it (and
    fp32 to float64) loses nothing, and the oracle computes from the very values the
    GPU reads."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    if a.dtype in (np.float32, np.float64):
        return a.astype(np.float64)
    raise TypeError(f"unsupported element type {a.dtype}")


def block_layout(L_in: int, sample_from_anchor: bool) -> tuple[int, int]:
    """(N, i_first_pred): prediction slots per block and the first predicting slot.

    [dflash-log], the paragraph saying that DSpark changes only the proposal: the block
    is anchor-first, slot 0 already predicts the first draft, so every one of the L_in
    slots predicts.
    [spec-pr], "Format differences": with sample_from_anchor false the block is the
    1+N infilling layout, slot 0 holds the bonus token and is not a prediction slot,
    so a block of 1+n_max slots yields n_max drafts; the read loop starts at
    i_first_pred = 1.
    """
    if sample_from_anchor:
        return L_in, 0
    if L_in < 2:
        raise ValueError("the 1+N layout needs at least two slots")
    return L_in - 1, 1


def base_logits(hidden, lm_head, lm_bias, i_first_pred: int, N: int,
                chunk: int = 8192) -> np.ndarray:
    """logits(i) = h[b, i_first_pred + i] . lm_head^T (+ lm_bias), shape [B, N, V].

    [dflash-log], the proposal formula: logits(i) is the plain lm_head projection of
    the slot's final hidden state (the projection DSpark corrects; [luce-pr]: it
    replaces the plain argmax projection).  [spec-pr], reduced draft vocab: rows the
    draft cannot produce get a -1e9 bias.  The oracle always evaluates every row of
    the vocabulary; masked rows simply carry their bias.  The vocabulary is walked in
    chunks only to bound memory.
    """
    h = upcast(hidden)                                   # [B, L_in, H]
    B, _, H = h.shape
    rows = h[:, i_first_pred:i_first_pred + N, :].reshape(B * N, H)
    lm_head = np.asarray(lm_head)
    V = lm_head.shape[0]
    z = np.empty((B * N, V), np.float64)
    wbuf = np.empty((min(chunk, V), H), np.float64)     # reused: avoids page faults
    for v0 in range(0, V, chunk):
        v1 = min(V, v0 + chunk)
        w = wbuf[:v1 - v0]
        if lm_head.dtype == np.uint16:
            w[...] = np.left_shift(lm_head[v0:v1], 16, dtype=np.uint32).view(np.float32)
        else:
            w[...] = lm_head[v0:v1]
        z[:, v0:v1] = rows @ w.T
    if lm_bias is not None:
        z += upcast(lm_bias)[None, :]
    return z.reshape(B, N, V)


def markov_bias(w1, w2_f64: np.ndarray, prev) -> np.ndarray:
    """markov_w2^T . markov_w1[prev]: the previous-token-conditioned rank-r logit bias.

    [dflash-log], the proposal formula.  ``prev`` may be a scalar or a vector of
    previous tokens (one per block); the result is [V] or [len(prev), V].
    ``w2_f64`` is markov_w2 [r, V] already upcast.
    """
    u = upcast(np.asarray(w1)[prev])                     # [r] or [B, r]
    return u @ w2_f64


def corrected_logits(z_row: np.ndarray, w1, w2_f64: np.ndarray, prev) -> np.ndarray:
    """logits'(i) = logits(i) + markov_w2^T . markov_w1[prev(i)]  ([dflash-log])."""
    return z_row + markov_bias(w1, w2_f64, prev)


def argmax_lowest(row: np.ndarray) -> int:
    """Index of the largest value; among equal maxima the lowest index.

    [dflash-log], the proposal formula: prev(i > 0) = argmax logits'(i - 1).  The pages
    do not say how ties break; the reading taken is the lowest token id."""
    m = row.max()
    return int(np.flatnonzero(row == m)[0])


def topk_sorted(row: np.ndarray, k: int) -> np.ndarray:
    """The k best indices of ``row`` by value descending, ties to the lower index.

    [ort-pr]: dspark_top_k is the number of candidates the lattice keeps per block
    slot; the order is this oracle's reading.
    """
    n = row.shape[-1]
    if k < n:
        # every member of the top k is >= the k-th largest value; sort only those
        kth = np.partition(row, n - k)[n - k]
        cand = np.flatnonzero(row >= kth)
    else:
        cand = np.arange(n)
    order = np.lexsort((cand, -row[cand]))
    return cand[order[:k]]


def confidence(hidden, w_conf, b_conf: float, i_first_pred: int, N: int) -> np.ndarray:
    """conf[b, i] = sigmoid(h[b, i_first_pred + i] . w_conf + b_conf), shape [B, N].

    [dflash-log], "spec: add confidence-based draft pruning for DSpark": the
    confidence head predicts each drafted position's acceptance.  Its form, a linear
    projection of the slot's hidden state followed by a logistic, is the reading that
    the head's name (conf_proj) and its use as the chance that a slot survives
    verification support.
    """
    h = upcast(hidden)[:, i_first_pred:i_first_pred + N, :]
    x = h @ upcast(w_conf) + float(b_conf)
    return 1.0 / (1.0 + np.exp(-x))


def truncation_length(conf_row: np.ndarray, conf_min: float) -> int:
    """Index of the first slot whose confidence is below conf_min, else N.

    [dflash-log], "spec: add confidence-based draft pruning for DSpark": the block ends
    at its first slot whose confidence falls under the threshold; a threshold of 0 (the
    default) turns the pruning off.
    "dflash: draft full n_max blocks ...": every block is drafted in full and
    truncated afterwards, so truncation only sets the length.
    """
    N = conf_row.shape[0]
    if conf_min <= 0.0:
        return N
    for i in range(N):
        if conf_row[i] < conf_min:
            return i
    return N


def greedy_chain(z_b: np.ndarray, w1, w2_f64: np.ndarray, anchor: int,
                 top_k: int = 1, topk_markov: bool = True):
    """The semi-autoregressive Markov-corrected greedy chain of one block.

    [dflash-log], the proposal formula: prev(0) is the block's anchor token and
    prev(i > 0) = argmax logits'(i - 1); the chain runs over the block's positions
    (and, on the pages, is vectorised across blocks).  [luce-pr]: the DDTree
    candidate top-k gets the Markov bias too (topk_markov=True); with
    topk_markov=False the candidates are ranked on the base logits.

    Returns (tok [N], topk_ids [N, k], topk_vals [N, k], zc [N, V]).
    """
    N, V = z_b.shape
    tok = np.empty(N, np.int64)
    ids = np.empty((N, top_k), np.int64)
    vals = np.empty((N, top_k), np.float64)
    zc = np.empty_like(z_b)
    prev = int(anchor)
    for i in range(N):
        zc[i] = corrected_logits(z_b[i], w1, w2_f64, prev)
        tok[i] = argmax_lowest(zc[i])
        ranked = zc[i] if topk_markov else z_b[i]
        ids[i] = topk_sorted(ranked, top_k)
        vals[i] = ranked[ids[i]]
        prev = int(tok[i])
    return tok, ids, vals, zc


def blank_past_cut(draft, tk_ids, tk_vals, n_draft) -> None:
    """Adaptive block length: the slots of block b from n_draft[b] on are not drafted
    (draft and top-k ids -1, top-k values NaN), in place.

    [dflash-log], "spec: add confidence-based draft pruning for DSpark": a block is cut
    at its first slot below the threshold and verify reads nothing past the cut.  The
    adaptive mode (a reading: the pages leave the wiring open) therefore drafts nothing
    there, and -1 / NaN mark the undrafted slots."""
    for b in range(draft.shape[0]):
        cut = int(n_draft[b])
        draft[b, cut:] = -1
        tk_ids[b, cut:] = -1
        tk_vals[b, cut:] = np.nan


def propose(hidden, anchors, lm_head, markov_w1, markov_w2, *, L_in: int,
            sample_from_anchor: bool, top_k: int, conf_min: float,
            lm_bias=None, w_conf=None, b_conf: float = 0.0,
            topk_markov: bool = True, return_logits: bool = False,
            skip_truncated: bool = False, conf_hidden=None) -> dict:
    """The whole proposal of a batch: base logits, chain, top-k, confidence, truncation.

    Returns a dict with draft [B, N], topk_ids / topk_vals [B, N, k], conf [B, N]
    (None without a confidence head), n_draft [B], base logits z [B, N, V] and, when
    asked, the corrected logits [B, N, V].

    ``skip_truncated``: the confidence-gated adaptive block length.  Truncation cuts a
    block at its first slot below conf_min ([dflash-log], confidence-based draft
    pruning) and verify reads nothing past that cut, so the slots after it need not be
    drafted at all: their draft and top-k ids read -1 and their top-k values NaN.  The
    slots before the cut, the confidences and n_draft are those of the full proposal.

    ``conf_hidden`` [B, L_in, H] (optional): [luce-pr], summary, names a calibrated
    confidence export taken before the final norm, i.e. a hidden state of its own for
    the confidence head.  When given, the confidence head reads it in place of
    ``hidden`` (same slots); the logits and the chain still read ``hidden``.
    """
    N, ifp = block_layout(L_in, sample_from_anchor)
    z = base_logits(hidden, lm_head, lm_bias, ifp, N)
    B = z.shape[0]
    w2 = upcast(markov_w2)
    draft = np.empty((B, N), np.int64)
    tk_ids = np.empty((B, N, top_k), np.int64)
    tk_vals = np.empty((B, N, top_k), np.float64)
    zc_all = np.empty_like(z) if return_logits else None
    anchors = np.asarray(anchors, np.int64)
    for b in range(B):
        tok, ids, vals, zc = greedy_chain(z[b], markov_w1, w2, int(anchors[b]),
                                          top_k, topk_markov)
        draft[b], tk_ids[b], tk_vals[b] = tok, ids, vals
        if return_logits:
            zc_all[b] = zc
    if w_conf is not None:
        conf = confidence(hidden if conf_hidden is None else conf_hidden, w_conf, b_conf,
                          ifp, N)
        n_draft = np.array([truncation_length(conf[b], conf_min) for b in range(B)],
                           np.int64)
    else:
        conf = None
        n_draft = np.full(B, N, np.int64)
    if skip_truncated:
        blank_past_cut(draft, tk_ids, tk_vals, n_draft)
    return dict(draft=draft, topk_ids=tk_ids, topk_vals=tk_vals, conf=conf,
                n_draft=n_draft, base_logits=z, logits=zc_all, N=N,
                i_first_pred=ifp)


def verify(draft, n_draft, target):
    """Greedy verify/accept, unchanged from DFlash.

    [dflash-log]: greedy stays lossless and the verify/accept path is DFlash's: the
    accepted length a is the longest prefix of the (truncated) draft equal to the
    target's argmax tokens, and the target's token at position a is the bonus token.
    ``target`` is [B, N+1]: the target's argmax after the anchor and after each
    drafted slot.  Returns (accepted [B], bonus [B], emitted [B, N+1]) where emitted
    holds draft[:a] followed by the bonus token and -1 after it.
    """
    draft = np.asarray(draft, np.int64)
    target = np.asarray(target, np.int64)
    B, N = draft.shape
    accepted = np.zeros(B, np.int64)
    bonus = np.zeros(B, np.int64)
    emitted = np.full((B, N + 1), -1, np.int64)
    for b in range(B):
        limit = min(max(int(n_draft[b]), 0), N)
        a = 0
        while a < limit and draft[b, a] == target[b, a]:
            a += 1
        accepted[b] = a
        bonus[b] = target[b, a]
        emitted[b, :a] = draft[b, :a]
        emitted[b, a] = bonus[b]
    return accepted, bonus, emitted


def tree_verify(topk_ids, n_draft, target):
    """Verify of the top-k candidate lattice (the DDTree consumer), greedy target.

    [luce-pr], description: the DDTree's candidates are the per-slot top-k, and they
    get the Markov bias too; its summary leaves the tree step itself unchanged.
    [ort-pr], the DFlash 2 and DSpark builder commits: a block drafter hands the runtime
    a lattice of dspark_top_k candidates per slot, which the runtime walks greedily, and
    DSpark reuses DFlash 2's verification path.  Reading (the pages define no tree
    construction): the tree is
    the whole lattice -- every candidate of slot i is a child of every candidate of slot
    i - 1 -- down to the truncated length n_draft[b].  The greedy target accepts the
    child equal to its own argmax after the accepted prefix; that prefix is always the
    target's own tokens, so its argmax at depth i is target[b, i].

    topk_ids [B, N, k], n_draft [B], target [B, N + 1].  Returns (accepted [B], bonus
    [B], emitted [B, N + 1], path [B, N]): accepted = the depth reached, bonus =
    target[b, accepted], emitted = the accepted tokens then the bonus then -1, path =
    the rank of the candidate taken at each accepted depth and -1 after.
    """
    ids = np.asarray(topk_ids, np.int64)
    target = np.asarray(target, np.int64)
    B, N, k = ids.shape
    accepted = np.zeros(B, np.int64)
    bonus = np.zeros(B, np.int64)
    emitted = np.full((B, N + 1), -1, np.int64)
    path = np.full((B, N), -1, np.int64)
    for b in range(B):
        limit = min(max(int(n_draft[b]), 0), N)
        depth = 0
        while depth < limit:
            rank = -1
            for q in range(k):
                if ids[b, depth, q] == target[b, depth]:
                    rank = q
                    break
            if rank < 0:
                break
            emitted[b, depth] = ids[b, depth, rank]
            path[b, depth] = rank
            depth += 1
        accepted[b] = depth
        bonus[b] = target[b, depth]
        emitted[b, depth] = bonus[b]
    return accepted, bonus, emitted, path
