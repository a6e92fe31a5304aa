"""The seeded input generators: determinism, shapes, the recipe's constraints."""
import numpy as np
import pytest
import torch

from workloads import WORKLOADS, Workload, make_batch, make_head, make_target, to_bf16_bits


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 3,
                        np.array([1.0, -2.5, 1 + 2 ** -8, 1 + 3 * 2 ** -9, 0.0], np.float32)])
    ours = to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_deterministic_and_shapes():
    wl = WORKLOADS["tiny_fp32"]
    h1, h2 = make_head(wl), make_head(wl)
    for k in ("lm_head", "markov_w1", "markov_w2", "w_conf"):
        assert np.array_equal(h1[k], h2[k])
    assert h1["lm_head"].shape == (wl.V, wl.H) and h1["lm_head"].dtype == np.float32
    assert h1["markov_w1"].shape == (wl.V, wl.r)
    assert h1["markov_w2"].shape == (wl.r, wl.V)
    b = make_batch(wl)
    assert b["hidden"].shape == (wl.B, wl.L_in, wl.H)
    assert b["anchors"].dtype == np.int32 and np.all((0 <= b["anchors"]) & (b["anchors"] < wl.V))
    assert abs(float(h1["lm_head"].std()) - wl.weight_std) < 0.002


def test_bf16_workload_bits():
    wl = WORKLOADS["qwen3_8b_b32"].scaled(V=1000, H=256, r=16)
    hd = make_head(wl)
    assert hd["lm_head"].dtype == np.uint16
    vals = (hd["lm_head"].astype(np.uint32) << 16).view(np.float32)
    assert abs(float(vals.std()) - 0.02) < 0.001


def test_mask_token_never_anchor():
    wl = WORKLOADS["qwen38_27b_b8"].scaled(B=20000, H=64, name="anchors-only")
    from workloads import _rng, _S_ANCHORS  # the same draw make_batch performs
    a = _rng(wl.seed, _S_ANCHORS).integers(0, wl.V - 1, size=wl.B)
    a = a + (a >= wl.mask_token)
    assert not np.any(a == wl.mask_token)
    assert a.max() < wl.V


def test_reduced_vocab_bias():
    wl = WORKLOADS["gemma4_bonus_b64"].scaled(V=5000, H=64, r=8, n_emit=300)
    hd = make_head(wl)
    assert hd["emit_rows"].shape == (300,)
    assert np.all(np.diff(hd["emit_rows"]) > 0)
    assert np.count_nonzero(hd["lm_bias"] == 0) == 300
    assert np.all(hd["lm_bias"][np.setdiff1d(np.arange(5000), hd["emit_rows"])] == -1e9)


@pytest.mark.parametrize("p", [None, 0.4])
def test_target_agreement(p):
    wl = WORKLOADS["qwen3_8b_b32"].scaled(accept_p=p, B=2000)
    rng = np.random.default_rng(1)
    draft = rng.integers(0, wl.V, (wl.B, wl.N))
    t = make_target(wl, draft)
    assert t.shape == (wl.B, wl.N + 1)
    agree = np.array([next((j for j in range(wl.N) if t[b, j] != draft[b, j]), wl.N)
                      for b in range(wl.B)])
    if p is None:
        assert np.all(agree < wl.N)
        assert abs(agree.mean() - (wl.N - 1) / 2) < 0.5
    else:
        # mean of min(Geom, N): sum_{j=1..N} (1-p)^j
        want = sum((1 - p) ** j for j in range(1, wl.N + 1))
        assert abs(agree.mean() - want) < 0.15
