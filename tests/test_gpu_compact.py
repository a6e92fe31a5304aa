"""A bias-form head (full-V lm_head + lm_bias masking rows) prepared in its compact form.

dspark_prepare_head finds the emittable rows on the device and gathers their weights;
the proposals then run on those rows only.  Checked here:
  * the prepared buffer's row list is the sorted emittable set (the documented layout);
  * the outputs match the oracle over the full head, for both chain forms' entry (the
    compact head is prepared, so the pruned chain runs) and both anchor layouts;
  * top_k above the emittable count: the call falls back to the full head, still right;
  * the kernel count and workspace size follow the compact head.
"""
import numpy as np
import pytest

from gpu_cases import compare, gpu_propose, oracle_run
from workloads import Workload, make_batch, make_head

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from dspark_block_drafter_gb300 import _abi  # noqa: E402
from dspark_block_drafter_gb300 import torch_io as tio  # noqa: E402


def _wl(**kw):
    base = dict(name="compact", B=6, L_in=5, H=128, V=4096, r=32, top_k=4,
                sample_from_anchor=True, conf_min=0.5, dtype="bf16", weight_std=0.2,
                conf_std=0.05, n_emit=300, seed=91)
    base.update(kw)
    return Workload(**base)


def _cfg(wl):
    return tio.make_config(wl.B, wl.L_in, wl.H, wl.V, wl.r, wl.top_k, wl.sample_from_anchor,
                           wl.conf_min, wl.dtype, wl.topk_markov)


def test_compact_row_list_is_the_emittable_set():
    wl = _wl(n_emit=301)                      # not a multiple of 8: padded to 304
    hd = make_head(wl)
    head = tio.head_to_device(hd).prepare(_cfg(wl))
    buf = head.prepared.cpu().numpy()
    hdr = buf[:256].view(np.int32)
    assert hdr[0] == 0x4D435044                # the compact header's magic
    V, H, r, n_emit, n_pad = hdr[1:6]
    assert (V, H, r, n_emit, n_pad) == (wl.V, wl.H, wl.r, 301, 304)
    rows = buf[256:256 + 4 * n_pad].view(np.int32)
    assert np.array_equal(rows[:n_emit], hd["emit_rows"])
    assert np.all(rows[n_emit:] == hd["emit_rows"][-1])


@pytest.mark.parametrize("sfa", [True, False])
@pytest.mark.parametrize("topk_markov", [True, False])
def test_compact_matches_oracle(sfa, topk_markov):
    wl = _wl(sample_from_anchor=sfa, topk_markov=topk_markov, L_in=6 if not sfa else 5)
    hd, bt = make_head(wl), make_batch(wl)
    g, _ = gpu_propose(wl, hd, bt, "full", chain="pruned")
    rep = compare(wl, hd, bt, oracle_run(wl, hd, bt), g, "full")
    assert rep["failures"] == [], rep
    emit = set(hd["emit_rows"].tolist())
    assert set(g["draft"].ravel().tolist()) <= emit
    assert set(g["topk_ids"].ravel().tolist()) <= emit


def test_topk_above_emittable_rows_uses_the_full_head():
    # k > n_emit: the call runs on the full head.  The ranks past the emittable rows hold
    # masked rows at bias -1e9, where fp32 cannot order them (-1e9 + z' rounds to -1e9:
    # they tie, and ties go to the lower row), so only what is defined is checked: the
    # draft and the emittable ranks equal the oracle's, the rest are masked rows.
    wl = _wl(n_emit=5, top_k=8)
    hd, bt = make_head(wl), make_batch(wl)
    g, _ = gpu_propose(wl, hd, bt, "full", chain="pruned")
    o = oracle_run(wl, hd, bt)
    emit = set(hd["emit_rows"].tolist())
    assert np.array_equal(g["draft"], o["draft"])
    assert np.array_equal(g["topk_ids"][..., :5], o["topk_ids"][..., :5])
    assert np.all(np.abs(g["topk_vals"][..., :5] - o["topk_vals"][..., :5]) <= 2e-2)
    assert not (set(g["topk_ids"][..., 5:].ravel().tolist()) & emit)
    assert np.all(g["topk_vals"][..., 5:] <= -1e8)


def test_kernel_count_follows_the_compact_head():
    wl = _wl(n_emit=256)
    hd = make_head(wl)
    cfg = _cfg(wl)
    prepared = tio.head_to_device(hd).prepare(cfg)
    out = tio.Outputs.allocate(wl.B, wl.N, wl.top_k, prepared.V_head)
    # the compact head, prepared: the pruned chain (reset, GEMM, tables)
    assert _abi.dspark_propose_kernel_count(cfg, prepared.struct(), out.struct()) == 3
    # top_k above the emittable rows: the full head's dense chain (reset, confidence,
    # GEMM, chain and the top-k merge)
    wl8 = _wl(n_emit=5, top_k=8)
    cfg8 = _cfg(wl8)
    p8 = tio.head_to_device(make_head(wl8)).prepare(cfg8)
    out8 = tio.Outputs.allocate(wl8.B, wl8.N, wl8.top_k, p8.V_head)
    assert _abi.dspark_propose_kernel_count(cfg8, p8.struct(), out8.struct()) == 5
