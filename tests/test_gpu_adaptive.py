"""Adaptive block length (skip_truncated): the GPU against the oracle, which blanks every
slot from a block's confidence cut on; the slots before it must match the full
proposal."""
import numpy as np
import pytest

from workloads import Workload, make_batch, make_head

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gpu_cases import gpu_propose, run_case  # noqa: E402


def _wl(**kw):
    base = dict(name="adaptive", B=32, L_in=16, H=128, V=2048, r=16, top_k=4,
                sample_from_anchor=True, conf_min=0.5, dtype="bf16", weight_std=0.2,
                conf_std=0.2, seed=616)
    base.update(kw)
    return Workload(**base)


@pytest.mark.parametrize("conf_min", [0.0, 0.3, 0.5, 0.9])
def test_adaptive_pair_tiles(conf_min):
    # 32 blocks x 16 slots: two 256-row N-tiles; at conf_min 0.9 nearly every block is
    # cut before slot 8, so the second N-tile is left out altogether
    g, o, rep = run_case(_wl(conf_min=conf_min), chain="pruned", skip_truncated=True)
    if conf_min == 0.0:
        assert (g["n_draft"] == 16).all() and (g["draft"] >= 0).all()
    if conf_min == 0.9:
        assert g["n_draft"].max() < 8 and (g["n_draft"] == 0).any()


@pytest.mark.parametrize("shape", [dict(B=64, L_in=7, sample_from_anchor=False),
                                   dict(B=3, L_in=5), dict(B=300, L_in=2),
                                   dict(B=2, L_in=40, conf_min=0.2)])
def test_adaptive_other_tilings(shape):
    run_case(_wl(**shape), chain="pruned", skip_truncated=True)


def test_adaptive_without_confidence_head():
    # no confidence head: nothing is cut
    wl = _wl()
    hd, bt = make_head(wl), make_batch(wl)
    hd["w_conf"] = None
    g, o, rep = run_case(wl, hd=hd, bt=bt, chain="pruned", skip_truncated=True)
    assert (g["n_draft"] == wl.N).all() and (g["draft"] >= 0).all()


def test_adaptive_prefix_equals_full_proposal():
    wl = _wl(conf_min=0.5)
    hd, bt = make_head(wl), make_batch(wl)
    full, _ = gpu_propose(wl, hd, bt, chain="pruned")
    cut, _ = gpu_propose(wl, hd, bt, chain="pruned", skip_truncated=True)
    assert np.array_equal(full["n_draft"], cut["n_draft"])
    for b in range(wl.B):
        c = int(cut["n_draft"][b])
        assert np.array_equal(cut["draft"][b, :c], full["draft"][b, :c])
        assert np.array_equal(cut["topk_ids"][b, :c], full["topk_ids"][b, :c])
        assert (cut["draft"][b, c:] == -1).all()


def test_adaptive_needs_the_pruned_chain():
    from dspark_block_drafter_gb300 import _abi
    wl = _wl()
    hd, bt = make_head(wl), make_batch(wl)
    with pytest.raises(_abi.DSparkError) as e:
        gpu_propose(wl, hd, bt, chain="dense", skip_truncated=True)
    assert e.value.status == _abi.DSPARK_ERR_UNSUPPORTED


@pytest.mark.parametrize("name", ["qwen3_8b_b32", "qwen38_27b_b8", "gemma4_bonus_b64"])
def test_adaptive_full_size(name):
    # the shapes the benchmark times, with work stopped at each block's confidence cut
    from workloads import WORKLOADS
    wl = WORKLOADS[name]
    g, o, rep = run_case(wl, chain="pruned", skip_truncated=True)
    assert (g["n_draft"] < wl.N).any()


def test_adaptive_every_block_cut_at_slot_zero():
    # every confidence is ~0: no block drafts anything, so the GEMM has no live N-tile
    # and no table CTA works; the walk still writes -1 / NaN everywhere
    g, o, rep = run_case(_wl(b_conf=-50.0), chain="pruned", skip_truncated=True)
    assert (g["n_draft"] == 0).all()
    assert (g["draft"] == -1).all() and (g["topk_ids"] == -1).all()
    assert np.isnan(g["topk_vals"]).all()
