"""Failure detection on the GPU without a fault: a bounded device-side wait that nothing
completes gives up, raises the timeout bit of the workspace error word, and the kernel
returns; the host reads DSPARK_ERR_TIMEOUT and the context keeps working."""
import pytest

from workloads import WORKLOADS

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import dspark_block_drafter_gb300 as ds  # noqa: E402
from dspark_block_drafter_gb300 import _abi, torch_io as tio  # noqa: E402
from gpu_cases import gpu_propose, run_case  # noqa: E402
from workloads import make_batch, make_head  # noqa: E402

MAX_SM_HZ = 2.07e9          # highest SM clock of the part: a budget cannot run out sooner


def _selftest(ws, budget, pre_abort=False):
    s = torch.cuda.current_stream()
    ds.check(ds.dspark_wait_selftest(ws.data_ptr(), ws.numel(), budget, pre_abort,
                                     s.cuda_stream))


def test_wait_runs_out_after_its_budget():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    _selftest(ws, 1000, pre_abort=True)                  # loads the module, not timed
    torch.cuda.synchronize()
    assert tio.device_status(ws) == _abi.DSPARK_ERR_TIMEOUT
    budget = 200_000_000
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    _selftest(ws, budget)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    # it waited the whole budget (no early return), and it did end
    assert ms >= 0.95 * budget / MAX_SM_HZ * 1e3, ms
    assert ms < 5000.0, ms
    assert tio.device_status(ws) == _abi.DSPARK_ERR_TIMEOUT
    # reading the status cleared it
    assert tio.device_status(ws) == _abi.DSPARK_OK


def test_abort_flag_ends_the_wait_at_once():
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    _selftest(ws, 1000, pre_abort=True)
    torch.cuda.synchronize()
    assert tio.device_status(ws) == _abi.DSPARK_ERR_TIMEOUT
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    _selftest(ws, 2_000_000_000, pre_abort=True)         # a 1 s budget, left at once
    e1.record()
    torch.cuda.synchronize()
    assert e0.elapsed_time(e1) < 100.0
    assert tio.device_status(ws) == _abi.DSPARK_ERR_TIMEOUT


def test_context_usable_after_a_timeout():
    # the timeout lands in a real proposal workspace; the next pass on that workspace
    # starts from a clear error word and matches the oracle
    wl = WORKLOADS["tiny_fp32"]
    hd, bt = make_head(wl), make_batch(wl)
    g, ws = gpu_propose(wl, hd, bt)
    _selftest(ws, 1_000_000)
    torch.cuda.synchronize()
    assert tio.device_status(ws) == _abi.DSPARK_ERR_TIMEOUT
    _selftest(ws, 1_000_000)
    cfg = tio.make_config(wl.B, wl.L_in, wl.H, wl.V, wl.r, wl.top_k, wl.sample_from_anchor,
                          wl.conf_min, wl.dtype, wl.topk_markov)
    head = tio.head_to_device(hd)
    out = tio.Outputs.allocate(wl.B, wl.N, wl.top_k, head.V_head)
    tio.propose(cfg, head, tio.to_device(bt["hidden"]), tio.to_device(bt["anchors"]), out,
                ws)
    torch.cuda.synchronize()
    assert tio.device_status(ws) == _abi.DSPARK_OK
    again = out.numpy()
    assert (again["draft"] == g["draft"]).all()
    run_case(wl)
