"""dspark_propose_noalloc: the proposal for callers that cannot allocate device memory.

Such callers (code running inside a host framework that owns every allocation, plugins
that must not touch the allocator) pass no workspace; the library uses its built-in
16 MiB device scratch instead.  These tests call the entry point through the C ABI and
check, on two calls in a row (the scratch keeps what the previous call left), that it
returns what dspark_propose with a caller workspace returns.

The scratch's error word is read with dspark_noalloc_device_status: a bad anchor is
reported there, and the next clean call reads clean.

This file is named so that pytest collects it last.
"""
import numpy as np
import pytest

from workloads import WORKLOADS, Workload, make_batch, make_head

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from dspark_block_drafter_gb300 import _abi  # noqa: E402
from dspark_block_drafter_gb300 import torch_io as tio  # noqa: E402

TOL = {"f32": 1e-5, "bf16": 2e-2}


def _setup(wl, prepared):
    hd, bt = make_head(wl), make_batch(wl)
    cfg = tio.make_config(wl.B, wl.L_in, wl.H, wl.V, wl.r, wl.top_k, wl.sample_from_anchor,
                          wl.conf_min, wl.dtype, wl.topk_markov)
    head = tio.head_to_device(hd)
    if prepared:
        head.prepare(cfg)
    return cfg, head, tio.to_device(bt["hidden"]), tio.to_device(bt["anchors"])


def _with_workspace(wl, cfg, head, hidden, anchors):
    out = tio.Outputs.allocate(wl.B, wl.N, wl.top_k, head.V_head)
    ws = tio.workspace_for(cfg, head)
    tio.propose(cfg, head, hidden, anchors, out, ws)
    torch.cuda.synchronize()
    return out.numpy()


def _no_alloc(wl, cfg, head, hidden, anchors):
    out = tio.Outputs.allocate(wl.B, wl.N, wl.top_k, head.V_head)
    # sentinel values: every output element must be written by the call
    for t in (out.draft, out.n_draft, out.topk_ids):
        t.fill_(-7)
    for t in (out.topk_vals, out.conf):
        t.fill_(float("nan"))
    _abi.check(_abi.dspark_propose_noalloc(cfg, head.struct(), hidden.data_ptr(),
                                           anchors.data_ptr(), out.struct(),
                                           torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return out.numpy()


def _same(ref, got, tol):
    for k in ("draft", "n_draft", "topk_ids"):
        assert np.array_equal(ref[k], got[k]), k
    for k in ("topk_vals", "conf"):
        assert np.all(np.abs(ref[k] - got[k]) <= tol), k


CASES = {
    "bf16-dense": (Workload("na", B=3, L_in=5, H=200, V=1000, r=24, top_k=5,
                            sample_from_anchor=True, conf_min=0.5, dtype="bf16",
                            weight_std=0.2, conf_std=0.05, seed=31), False),
    "bf16-pruned-1+N": (Workload("na", B=4, L_in=7, H=256, V=2048, r=32, top_k=3,
                                 sample_from_anchor=False, conf_min=0.5, dtype="bf16",
                                 weight_std=0.1, conf_std=0.05, seed=32), True),
    "fp32-tiny": (WORKLOADS["tiny_fp32"], False),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_no_alloc_matches_workspace_path_twice(case):
    wl, prepared = CASES[case]
    cfg, head, hidden, anchors = _setup(wl, prepared)
    ref = _with_workspace(wl, cfg, head, hidden, anchors)
    first = _no_alloc(wl, cfg, head, hidden, anchors)
    second = _no_alloc(wl, cfg, head, hidden, anchors)
    _same(ref, first, TOL[wl.dtype])
    _same(ref, second, TOL[wl.dtype])


def test_no_alloc_rejects_calls_beyond_its_scratch():
    # the Qwen3-8B-shaped B=32 head needs far more than 16 MiB of scratch: refused on the
    # host, before anything is launched
    wl = WORKLOADS["qwen3_8b_b32"]
    cfg = tio.make_config(wl.B, wl.L_in, wl.H, wl.V, wl.r, wl.top_k, True, wl.conf_min, "bf16")
    head = _abi.dspark_head(lm_head=0x10000, V_head=wl.V, markov_w1=0x20000,
                            markov_w2=0x30000)
    out = _abi.dspark_outputs(draft=0x100, n_draft=0x200)
    st = _abi.dspark_propose_noalloc(cfg, head, 0x40000, 0x50000, out, 0)
    assert st == _abi.DSPARK_ERR_WORKSPACE
    assert "16777216" in _abi.dspark_last_error()


@pytest.mark.parametrize("case", ["bf16-dense", "bf16-pruned-1+N"])
def test_no_alloc_device_errors_are_readable(case):
    wl, prepared = CASES[case]
    cfg, head, hidden, anchors = _setup(wl, prepared)
    stream = torch.cuda.current_stream().cuda_stream
    bad = anchors.clone()
    bad[1] = wl.V + 3                            # a token outside [0, V)
    out = tio.Outputs.allocate(wl.B, wl.N, wl.top_k, head.V_head)
    _abi.check(_abi.dspark_propose_noalloc(cfg, head.struct(), hidden.data_ptr(),
                                           bad.data_ptr(), out.struct(), stream))
    assert _abi.dspark_noalloc_device_status(stream) == _abi.DSPARK_ERR_DEVICE
    assert "outside" in _abi.dspark_last_error()
    assert _abi.dspark_noalloc_device_status(stream) == _abi.DSPARK_OK   # read clears it
    # a bad call, then a good one: the good call starts from a clear word
    _abi.check(_abi.dspark_propose_noalloc(cfg, head.struct(), hidden.data_ptr(),
                                           bad.data_ptr(), out.struct(), stream))
    ref = _with_workspace(wl, cfg, head, hidden, anchors)
    got = _no_alloc(wl, cfg, head, hidden, anchors)
    assert _abi.dspark_noalloc_device_status(stream) == _abi.DSPARK_OK
    _same(ref, got, TOL[wl.dtype])
