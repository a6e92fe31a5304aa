"""The tolerance checker flags wrong results and accepts legal near-tie choices."""
import numpy as np

from oracle import check, propose


def _case(seed=3, near_tie=False):
    rng = np.random.default_rng(seed)
    B, L, H, V, r, k = 3, 5, 16, 200, 4, 3
    hidden = rng.standard_normal((B, L, H)).astype(np.float32)
    W = rng.standard_normal((V, H)).astype(np.float32)
    if near_tie:
        W[7] = W[11] * np.float32(1.0 + 1e-4)   # rows 7 and 11 nearly equal
    w1 = (rng.standard_normal((V, r)) * 0.3).astype(np.float32)
    w2 = (rng.standard_normal((r, V)) * 0.3).astype(np.float32)
    wc = rng.standard_normal(H).astype(np.float32)
    anchors = rng.integers(0, V, B)
    o = propose(hidden, anchors, W, w1, w2, L_in=L, sample_from_anchor=True, top_k=k,
                conf_min=0.5, w_conf=wc, return_logits=True)
    gpu = dict(draft=o["draft"].copy(), topk_ids=o["topk_ids"].copy(),
               topk_vals=o["topk_vals"].astype(np.float32), conf=o["conf"].astype(np.float32),
               n_draft=o["n_draft"].copy(), logits=o["logits"].astype(np.float32))
    kw = dict(anchors=anchors, markov_w1=w1, markov_w2=w2, top_k=k, topk_markov=True,
              conf_min=0.5, tol=2e-2)
    return o, gpu, kw


def test_exact_copy_passes():
    o, gpu, kw = _case()
    rep = check.check_propose(o, gpu=gpu, **kw)
    assert rep["failures"] == []


def test_wrong_token_flagged():
    o, gpu, kw = _case()
    gpu["draft"][1, 2] = (gpu["draft"][1, 2] + 1) % 200
    assert check.check_propose(o, gpu=gpu, **kw)["failures"]


def test_wrong_topk_flagged():
    o, gpu, kw = _case()
    gpu["topk_ids"][0, 1, [1, 2]] = gpu["topk_ids"][0, 1, [2, 1]]
    gpu["topk_vals"][0, 1, [1, 2]] = gpu["topk_vals"][0, 1, [2, 1]]
    rep = check.check_propose(o, gpu=gpu, **kw)
    z = o["logits"][0, 1]
    ids = o["topk_ids"][0, 1]
    if abs(z[ids[1]] - z[ids[2]]) > 2e-2:
        assert rep["failures"]


def test_conf_and_ndraft_flagged():
    o, gpu, kw = _case()
    gpu["conf"][0, 0] += 0.1
    assert check.check_propose(o, gpu=gpu, **kw)["failures"]
    o, gpu, kw = _case()
    gpu["n_draft"][2] = (gpu["n_draft"][2] + 1) % 6
    assert check.check_propose(o, gpu=gpu, **kw)["failures"]


def test_logits_flagged():
    o, gpu, kw = _case()
    gpu["logits"][2, 3, 17] += 0.05
    assert check.check_propose(o, gpu=gpu, **kw)["failures"]


def test_near_tie_alternative_accepted_and_chain_followed():
    # force a near tie at one slot by construction: pick the GPU's token as the
    # runner-up whenever the oracle margin is below tol
    o, gpu, kw = _case()
    z = o["logits"]
    found = False
    for b in range(z.shape[0]):
        s = np.sort(z[b, 0])
        if s[-1] - s[-2] < 5.0:
            # pretend the tolerance is wide enough for this pair to be a near tie
            kw2 = dict(kw, tol=float(s[-1] - s[-2]) + 1e-9)
            alt = int(np.flatnonzero(z[b, 0] == s[-2])[0])
            gpu2 = {k: (v.copy() if v is not None else None) for k, v in gpu.items()}
            gpu2.pop("logits")
            gpu2.pop("topk_ids")
            gpu2.pop("topk_vals")
            gpu2["draft"][b, 0] = alt
            # the rest of the GPU chain follows the alternative token
            from oracle import dspark_oracle as O
            w2 = O.upcast(kw["markov_w2"])
            prev = alt
            for i in range(1, z.shape[1]):
                zc = O.corrected_logits(o["base_logits"][b, i], kw["markov_w1"], w2, prev)
                gpu2["draft"][b, i] = O.argmax_lowest(zc)
                prev = gpu2["draft"][b, i]
            rep = check.check_propose(o, gpu=gpu2, **kw2)
            assert rep["failures"] == [], rep
            found = True
            break
    assert found


def test_verify_check():
    d = np.array([[1, 2, 3]])
    t = np.array([[1, 2, 0, 5]])
    assert check.check_verify(d, [3], t, [2], [0]) == []
    assert check.check_verify(d, [3], t, [3], [0])


def test_masked_rows_only_need_to_stay_masked():
    rng = np.random.default_rng(4)
    B, L, H, V, r, k = 2, 4, 16, 150, 4, 2
    hidden = rng.standard_normal((B, L, H)).astype(np.float32)
    W = rng.standard_normal((V, H)).astype(np.float32)
    w1 = (rng.standard_normal((V, r)) * 0.3).astype(np.float32)
    w2 = (rng.standard_normal((r, V)) * 0.3).astype(np.float32)
    bias = np.zeros(V, np.float32)
    bias[::3] = -1e9
    anchors = rng.integers(0, V, B)
    o = propose(hidden, anchors, W, w1, w2, L_in=L, sample_from_anchor=True, top_k=k,
                conf_min=0.0, lm_bias=bias, return_logits=True)
    # fp32-sized error on the masked rows only
    logits = (o["logits"] + np.where(bias < 0, 30.0, 0.0)).astype(np.float32)
    g = dict(draft=o["draft"], n_draft=o["n_draft"], logits=logits)
    kw = dict(anchors=anchors, markov_w1=w1, markov_w2=w2, top_k=k, topk_markov=True,
              conf_min=0.0, tol=2e-2, lm_bias=bias)
    assert check.check_propose(o, gpu=g, **kw)["failures"] == []
    logits[0, 0, 0] = 0.0            # a masked row that came back unmasked
    rep = check.check_propose(o, gpu=g, **kw)
    assert any("mask" in f for f in rep["failures"])
    logits[0, 0, 0] = -1e9
    logits[1, 2, 1] += 0.1           # an emittable row off by more than tol
    rep = check.check_propose(o, gpu=g, **kw)
    assert any("off by" in f for f in rep["failures"])


def _adaptive(gpu, o):
    # the GPU's adaptive output: blanked past the (oracle's) cut
    from oracle import dspark_oracle as O
    g = {k: (None if v is None else np.array(v)) for k, v in gpu.items() if k != "logits"}
    g["topk_vals"] = g["topk_vals"].astype(np.float32)
    O.blank_past_cut(g["draft"], g["topk_ids"], g["topk_vals"], g["n_draft"])
    return g


def test_adaptive_block_length_passes_and_flags():
    o, gpu, kw = _case(seed=8)
    assert (o["n_draft"] < 5).any()                 # some block is cut
    g = _adaptive(gpu, o)
    assert check.check_propose(o, gpu=g, skip_truncated=True, **kw)["failures"] == []
    # the same output checked as a full proposal fails (slots past the cut read -1)
    assert check.check_propose(o, gpu=g, **kw)["failures"]
    b = int(np.flatnonzero(o["n_draft"] < 5)[0])
    cut = int(o["n_draft"][b])
    bad = {k: v.copy() for k, v in g.items()}
    bad["draft"][b, cut] = 3                        # a token past the cut
    assert check.check_propose(o, gpu=bad, skip_truncated=True, **kw)["failures"]
    bad = {k: v.copy() for k, v in g.items()}
    bad["topk_vals"][b, cut, 0] = 1.0               # a value past the cut
    assert check.check_propose(o, gpu=bad, skip_truncated=True, **kw)["failures"]
    if cut > 0:
        bad = {k: v.copy() for k, v in g.items()}
        bad["draft"][b, cut - 1] = -1               # a slot before the cut left blank
        assert check.check_propose(o, gpu=bad, skip_truncated=True, **kw)["failures"]


def test_topk_values_alone_flagged():
    # ids right, one value off by more than the tolerance
    o, gpu, kw = _case()
    gpu["topk_vals"][1, 0, 2] += np.float32(0.05)
    assert check.check_propose(o, gpu=gpu, **kw)["failures"]
    o, gpu, kw = _case()
    gpu["topk_vals"][1, 0, 2] += np.float32(0.005)        # within tolerance
    assert check.check_propose(o, gpu=gpu, **kw)["failures"] == []


def test_invalid_topk_ids_flagged():
    for bad in ("duplicate", "negative", "too_large"):
        o, gpu, kw = _case()
        ids = gpu["topk_ids"][2, 4]
        if bad == "duplicate":
            ids[2] = ids[0]
        elif bad == "negative":
            ids[1] = -1
        else:
            ids[0] = 200
        rep = check.check_propose(o, gpu=gpu, **kw)
        assert any("invalid" in f for f in rep["failures"]), bad


def test_draft_out_of_range_flagged():
    o, gpu, kw = _case()
    gpu["draft"][0, 3] = 200
    assert any("out of range" in f for f in check.check_propose(o, gpu=gpu, **kw)["failures"])


def test_verify_emitted_flagged():
    rng = np.random.default_rng(5)
    draft = rng.integers(0, 9, (4, 5))
    n_draft = np.array([5, 3, 0, 5])
    target = draft.copy()
    target = np.concatenate([target, rng.integers(0, 9, (4, 1))], axis=1)
    target[3, 2] = (target[3, 2] + 1) % 9
    from oracle import verify
    a, b, e = verify(draft, n_draft, target)
    assert check.check_verify(draft, n_draft, target, a, b, e) == []
    e2 = e.copy()
    e2[0, 0] = (e2[0, 0] + 1) % 9
    assert check.check_verify(draft, n_draft, target, a, b, e2)
    b2 = b.copy()
    b2[1] = (b2[1] + 1) % 9
    assert check.check_verify(draft, n_draft, target, a, b2, e)
