"""Tolerance checker: compares a GPU proposal/verify result with the oracle.

TEST INFRASTRUCTURE ONLY.

The rule (stated with the method's requirements for this build):
  * logits, top-k values and confidences lie within ``tol`` (absolute) of the oracle;
  * a draft token is bit-exact wherever the oracle's top-1/top-2 margin of the
    corrected logits exceeds ``tol``; elsewhere the chosen token's oracle logit lies
    within ``tol`` of the oracle's maximum;
  * top-k ids are bit-exact wherever every adjacent gap among the oracle's best k+1
    values exceeds ``tol``; elsewhere each reported id's oracle value lies within
    ``tol`` of the oracle's value at the same rank;
  * n_draft is bit-exact wherever no confidence up to the oracle's cut lies within
    ``tol`` of conf_min, and always equals the first slot where the GPU's own
    confidence is below conf_min;
  * verify outputs are exact integers.

Teacher forcing: the check walks the GPU's chain.  After a slot whose GPU token was
accepted as a legal near-tie choice, the oracle's next slot is evaluated with that
token as prev, so one legal divergence cannot cascade into false failures.  A token
is only ever fed back after it has passed the check above.
"""
from __future__ import annotations

import numpy as np

from .dspark_oracle import (MASK_BIAS_LIMIT, argmax_lowest, corrected_logits, topk_sorted,
                            upcast, verify)


def check_propose(oracle_out: dict, *, anchors, markov_w1, markov_w2, top_k: int,
                  topk_markov: bool, conf_min: float, gpu: dict, tol: float,
                  head_rows=None, lm_bias=None, max_report: int = 20,
                  skip_truncated: bool = False) -> dict:
    """Compare GPU proposal outputs with the oracle.

    ``oracle_out`` is the dict of :func:`oracle.propose` (its base logits are used).
    ``gpu`` holds numpy arrays draft [B,N], n_draft [B] and optionally topk_ids,
    topk_vals [B,N,k], conf [B,N], logits [B,N,V or V_head].
    ``head_rows`` maps the GPU's logits columns to token ids when the GPU evaluated a
    compact head (d2t form); None means the columns are the token ids.
    ``lm_bias`` (the full-vocabulary bias, or None) marks masked rows: their logits are
    about -1e9, where fp32 spacing is 64, so for them the check is only that the GPU
    value stays at or below the mask limit.
    ``skip_truncated``: the GPU ran the adaptive block length.  Slots before the GPU's
    own n_draft[b] are checked as usual (n_draft itself as below); after it, the draft
    and top-k ids must read -1 and the top-k values NaN.
    Returns {"failures": [...], "near_ties": int, "slots": int}.
    """
    z = oracle_out["base_logits"]
    B, N, V = z.shape
    w2 = upcast(markov_w2)
    fails: list[str] = []
    near = 0
    masked = None if lm_bias is None else upcast(lm_bias) <= MASK_BIAS_LIMIT

    def fail(msg):
        if len(fails) < max_report:
            fails.append(msg)

    g_draft = np.asarray(gpu["draft"]).astype(np.int64)
    g_ids = gpu.get("topk_ids")
    g_vals = gpu.get("topk_vals")
    g_logits = gpu.get("logits")
    g_nd = np.asarray(gpu["n_draft"]).astype(np.int64)
    for b in range(B):
        prev = int(anchors[b])
        for i in range(N):
            if skip_truncated and i >= g_nd[b]:
                # past the cut: nothing drafted
                if int(g_draft[b, i]) != -1:
                    fail(f"draft[{b},{i}]={int(g_draft[b, i])} past n_draft={g_nd[b]}, not -1")
                if g_ids is not None and np.any(np.asarray(g_ids[b, i]) != -1):
                    fail(f"topk_ids[{b},{i}] past n_draft={g_nd[b]} not all -1")
                if g_vals is not None and not np.all(np.isnan(np.asarray(g_vals[b, i]))):
                    fail(f"topk_vals[{b},{i}] past n_draft={g_nd[b]} not all NaN")
                continue
            zc = corrected_logits(z[b, i], markov_w1, w2, prev)
            g = int(g_draft[b, i])
            if not 0 <= g < V:
                fail(f"draft[{b},{i}]={g} out of range")
                break
            best = argmax_lowest(zc)
            top2 = np.partition(zc, V - 2)[-2:] if V >= 2 else np.array([-np.inf, zc[0]])
            margin = top2[1] - top2[0]
            if margin > tol:
                if g != best:
                    fail(f"draft[{b},{i}]={g} but oracle argmax {best} "
                         f"(margin {margin:.3g} > tol)")
            else:
                near += 1
                if zc[g] < zc[best] - tol:
                    fail(f"draft[{b},{i}]={g}: logit {zc[g]:.6g} below max "
                         f"{zc[best]:.6g} - tol")
            ranked = zc if topk_markov else z[b, i]
            if g_ids is not None:
                ids = np.asarray(g_ids[b, i]).astype(np.int64)
                kk = min(top_k + 1, V)
                o_ids = topk_sorted(ranked, kk)
                o_vals = ranked[o_ids]
                if np.any(ids < 0) or np.any(ids >= V) or len(set(ids.tolist())) != top_k:
                    fail(f"topk_ids[{b},{i}] invalid: {ids}")
                else:
                    gaps = -np.diff(o_vals)
                    if np.all(gaps > tol):
                        if not np.array_equal(ids, o_ids[:top_k]):
                            fail(f"topk_ids[{b},{i}]={ids} != oracle {o_ids[:top_k]}")
                    else:
                        dev = np.abs(ranked[ids] - o_vals[:top_k])
                        if np.any(dev > tol):
                            fail(f"topk_ids[{b},{i}]={ids}: rank values off by "
                                 f"{dev.max():.3g}")
                    if g_vals is not None:
                        dv = np.abs(np.asarray(g_vals[b, i], np.float64) - ranked[ids])
                        if np.any(dv > tol):
                            fail(f"topk_vals[{b},{i}] off by {dv.max():.3g}")
            if g_logits is not None:
                gl = np.asarray(g_logits[b, i], np.float64)
                ref = zc if head_rows is None else zc[head_rows]
                d = np.abs(gl - ref)
                if masked is not None:
                    mcols = masked if head_rows is None else masked[head_rows]
                    d[mcols] = 0.0
                    if np.any(gl[mcols] > MASK_BIAS_LIMIT):
                        fail(f"logits[{b},{i}]: a masked row rose above the mask limit")
                if np.any(d > tol):
                    j = int(np.argmax(d))
                    fail(f"logits[{b},{i}] off by {d[j]:.3g} at column {j}")
            prev = g
    # confidence and truncation
    o_conf = oracle_out.get("conf")
    g_conf = gpu.get("conf")
    if o_conf is not None and g_conf is not None:
        g_conf = np.asarray(g_conf, np.float64)
        d = np.abs(g_conf - o_conf)
        if np.any(d > tol):
            fail(f"conf off by {d.max():.3g}")
        for b in range(B):
            own = N
            if conf_min > 0:
                below = np.flatnonzero(np.asarray(gpu["conf"][b]) < np.float32(conf_min))
                own = int(below[0]) if below.size else N
            if g_nd[b] != own:
                fail(f"n_draft[{b}]={g_nd[b]} inconsistent with GPU conf (first below: {own})")
            o_nd = int(oracle_out["n_draft"][b])
            span = o_conf[b, :min(o_nd + 1, N)]
            if conf_min <= 0 or np.all(np.abs(span - conf_min) > tol):
                if g_nd[b] != o_nd:
                    fail(f"n_draft[{b}]={g_nd[b]} != oracle {o_nd}")
    else:
        for b in range(B):
            if g_nd[b] != oracle_out["n_draft"][b]:
                fail(f"n_draft[{b}]={g_nd[b]} != oracle {oracle_out['n_draft'][b]}")
    return {"failures": fails, "near_ties": near, "slots": B * N}


def check_verify(draft, n_draft, target, accepted, bonus, emitted=None) -> list[str]:
    """Exact comparison of a GPU verify result with the oracle on the same inputs."""
    a, bo, em = verify(draft, n_draft, target)
    fails = []
    if not np.array_equal(np.asarray(accepted, np.int64), a):
        fails.append(f"accepted {np.asarray(accepted)} != oracle {a}")
    if not np.array_equal(np.asarray(bonus, np.int64), bo):
        fails.append(f"bonus {np.asarray(bonus)} != oracle {bo}")
    if emitted is not None and not np.array_equal(np.asarray(emitted, np.int64), em):
        fails.append("emitted differs from oracle")
    return fails
