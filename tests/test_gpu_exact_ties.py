"""Bit-exact parity with ties: small-integer weights and hidden states make every product
and sum exact in bf16 operands with fp32 accumulation, so the GPU's corrected logits are
the oracle's exactly.  Drafts, top-k ids and top-k values must then equal the oracle's
with no tolerance, including the lowest-id rule wherever values tie."""
import numpy as np
import pytest

from oracle import propose as oracle_propose
from workloads import Workload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gpu_cases import gpu_propose  # noqa: E402


def _bf16_bits(a):
    # small integers have no low mantissa bits, so the bf16 pattern is exact
    return (np.ascontiguousarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _integer_case(seed, B, L_in, sfa, topk_markov, H=64, V=1024, r=8, k=4):
    rng = np.random.default_rng(seed)

    def ints(*shape):
        return rng.integers(-2, 3, size=shape).astype(np.float32)

    wl = Workload("int_ties", B=B, L_in=L_in, H=H, V=V, r=r, top_k=k, sample_from_anchor=sfa,
                  conf_min=0.0, dtype="bf16", weight_std=1.0, conf_std=1.0,
                  topk_markov=topk_markov, seed=seed)
    hd = dict(lm_head=_bf16_bits(ints(V, H)), markov_w1=_bf16_bits(ints(V, r)),
              markov_w2=_bf16_bits(ints(r, V)), w_conf=None, b_conf=0.0, lm_bias=None,
              emit_rows=None)
    bt = dict(hidden=_bf16_bits(ints(B, L_in, H)),
              anchors=rng.integers(0, V, size=B).astype(np.int32))
    return wl, hd, bt


@pytest.mark.parametrize("chain,B,L_in,sfa,topk_markov", [
    ("pruned", 32, 8, True, True),      # pair tiles of 256 prediction rows
    ("dense", 32, 8, True, True),
    ("pruned", 16, 5, False, True),     # 1+N layout
    ("dense", 16, 5, False, False),     # top-k over the base logits
    ("pruned", 8, 4, True, False),
])
def test_integer_logits_bit_exact(chain, B, L_in, sfa, topk_markov):
    wl, hd, bt = _integer_case(4242 + B + L_in, B, L_in, sfa, topk_markov)
    g, _ = gpu_propose(wl, hd, bt, chain=chain)
    o = oracle_propose(bt["hidden"], bt["anchors"], hd["lm_head"], hd["markov_w1"],
                       hd["markov_w2"], L_in=wl.L_in, sample_from_anchor=sfa,
                       top_k=wl.top_k, conf_min=0.0, topk_markov=topk_markov)
    # the case must actually contain ties for the rule to be tested
    zc_rows = o["topk_vals"].reshape(-1, wl.top_k)
    assert np.any(zc_rows[:, :-1] == zc_rows[:, 1:])
    assert np.array_equal(g["draft"], o["draft"])
    assert np.array_equal(g["topk_ids"], o["topk_ids"])
    assert np.array_equal(g["topk_vals"].astype(np.float64), o["topk_vals"])
    assert (g["n_draft"] == wl.N).all()


def _ternary_bits(rng, shape, p_nonzero):
    """bf16 bit patterns of values in {-1, 0, 1}, each nonzero with p_nonzero (split
    evenly between the signs)."""
    u = rng.random(shape, dtype=np.float32)
    bits = np.zeros(shape, np.uint16)
    bits[u < p_nonzero / 2] = 0x3F80                          # +1.0
    bits[(u >= p_nonzero / 2) & (u < p_nonzero)] = 0xBF80     # -1.0
    return bits


def test_integer_logits_bit_exact_full_size():
    # the Qwen3-8B-shaped head at B=32 that the benchmark times, through both chains:
    # |z| <= H = 4096 and |Markov term| <= r = 256 stay exact in fp32; sparse Markov
    # weights keep the pruning bound as tight as on the benchmark's inputs
    B, L_in, H, V, r, k = 32, 16, 4096, 151936, 256, 8
    rng = np.random.default_rng(777)
    wl = Workload("int_ties_full", B=B, L_in=L_in, H=H, V=V, r=r, top_k=k,
                  sample_from_anchor=True, conf_min=0.0, dtype="bf16", weight_std=1.0,
                  conf_std=1.0, seed=777)
    hd = dict(lm_head=_ternary_bits(rng, (V, H), 0.5),
              markov_w1=_ternary_bits(rng, (V, r), 0.05),
              markov_w2=_ternary_bits(rng, (r, V), 0.05), w_conf=None, b_conf=0.0,
              lm_bias=None, emit_rows=None)
    bt = dict(hidden=_ternary_bits(rng, (B, L_in, H), 0.5),
              anchors=rng.integers(0, V, size=B).astype(np.int32))
    o = oracle_propose(bt["hidden"], bt["anchors"], hd["lm_head"], hd["markov_w1"],
                       hd["markov_w2"], L_in=L_in, sample_from_anchor=True, top_k=k,
                       conf_min=0.0)
    vals = o["topk_vals"].reshape(-1, k)
    assert np.any(vals[:, :-1] == vals[:, 1:])
    for chain in ("pruned", "dense"):
        g, _ = gpu_propose(wl, hd, bt, chain=chain)
        assert np.array_equal(g["draft"], o["draft"]), chain
        assert np.array_equal(g["topk_ids"], o["topk_ids"]), chain
        assert np.array_equal(g["topk_vals"].astype(np.float64), o["topk_vals"]), chain


@pytest.mark.parametrize("name", ["qwen38_27b_b8", "gemma4_bonus_b64"])
def test_integer_logits_bit_exact_other_full_sizes(name):
    # the other large shapes: a 5120-wide head over 248320 rows at B=8, and the 1+N layout
    # over 262144 rows of which 32768 are emittable (both reduced-vocabulary forms)
    from workloads import WORKLOADS
    base = WORKLOADS[name]
    wl = Workload("int_" + name, B=base.B, L_in=base.L_in, H=base.H, V=base.V, r=base.r,
                  top_k=base.top_k, sample_from_anchor=base.sample_from_anchor,
                  conf_min=0.0, dtype="bf16", weight_std=1.0, conf_std=1.0,
                  n_emit=base.n_emit, seed=778)
    rng = np.random.default_rng(778)
    hd = dict(lm_head=_ternary_bits(rng, (wl.V, wl.H), 0.5),
              markov_w1=_ternary_bits(rng, (wl.V, wl.r), 0.05),
              markov_w2=_ternary_bits(rng, (wl.r, wl.V), 0.05), w_conf=None, b_conf=0.0,
              lm_bias=None, emit_rows=None)
    forms = ["full"]
    if wl.n_emit:
        emit = np.sort(rng.choice(wl.V, size=wl.n_emit, replace=False)).astype(np.int32)
        hd["lm_bias"] = np.full(wl.V, -1e9, np.float32)
        hd["lm_bias"][emit] = 0.0
        hd["emit_rows"] = emit
        forms.append("d2t")
    bt = dict(hidden=_ternary_bits(rng, (wl.B, wl.L_in, wl.H), 0.5),
              anchors=rng.integers(0, wl.V, size=wl.B).astype(np.int32))
    o = oracle_propose(bt["hidden"], bt["anchors"], hd["lm_head"], hd["markov_w1"],
                       hd["markov_w2"], L_in=wl.L_in, sample_from_anchor=wl.sample_from_anchor,
                       top_k=wl.top_k, conf_min=0.0, lm_bias=hd["lm_bias"])
    if wl.top_k > 1:
        vals = o["topk_vals"].reshape(-1, wl.top_k)
        assert np.any(vals[:, :-1] == vals[:, 1:])
    for form in forms:
        for chain in ("pruned", "dense"):
            g, _ = gpu_propose(wl, hd, bt, form, chain=chain)
            assert np.array_equal(g["draft"], o["draft"]), (form, chain)
            assert np.array_equal(g["topk_ids"], o["topk_ids"]), (form, chain)
            assert np.array_equal(g["topk_vals"].astype(np.float64), o["topk_vals"]), \
                (form, chain)
