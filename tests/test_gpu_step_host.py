"""dspark_step_host (host buffers in, host buffers out) against the device-pointer path
and the oracle's verify, with page-locked host buffers (read and written in place by the
kernels) and with pageable ones (copied through workspace staging)."""
import numpy as np
import pytest

from workloads import Workload, make_batch, make_conf_hidden, make_head, make_target

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gpu_cases import gpu_propose  # noqa: E402
from oracle import verify as oracle_verify  # noqa: E402


def _wl(**kw):
    base = dict(name="step_host", B=32, L_in=8, H=256, V=2048, r=32, top_k=4,
                sample_from_anchor=True, conf_min=0.5, dtype="bf16", weight_std=0.2,
                conf_std=0.05, accept_p=0.4, seed=515)
    base.update(kw)
    return Workload(**base)


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("chain", ["dense", "pruned"])
@pytest.mark.parametrize("with_topk", [True, False])
@pytest.mark.parametrize("conf_input", [False, True])
def test_step_host_matches_device_path(pinned, chain, with_topk, conf_input):
    from dspark_block_drafter_gb300 import _abi
    from dspark_block_drafter_gb300 import torch_io as tio
    wl = _wl()
    hd, bt = make_head(wl), make_batch(wl)
    ch = make_conf_hidden(wl) if conf_input else None
    g, _ = gpu_propose(wl, hd, bt, chain=chain, conf_hidden=ch)
    target = make_target(wl, g["draft"]).astype(np.int32)

    cfg = tio.make_config(wl.B, wl.L_in, wl.H, wl.V, wl.r, wl.top_k, wl.sample_from_anchor,
                          wl.conf_min, wl.dtype, wl.topk_markov)
    head = tio.head_to_device(hd)
    if chain == "pruned":
        head.prepare(cfg)
    B, N, k = wl.B, wl.N, wl.top_k

    def host(t):
        return t.pin_memory() if pinned else t

    hidden_h = host(tio.to_device(bt["hidden"], "cpu").contiguous())
    ch_h = host(tio.to_device(ch, "cpu").contiguous()) if conf_input else None
    anchors_h = host(torch.from_numpy(np.ascontiguousarray(bt["anchors"], dtype=np.int32)))
    target_h = host(torch.from_numpy(np.ascontiguousarray(target)))
    i32 = dict(dtype=torch.int32)
    draft_h, nd_h = host(torch.full((B, N), -7, **i32)), host(torch.full((B,), -7, **i32))
    acc_h, bon_h = host(torch.full((B,), -7, **i32)), host(torch.full((B,), -7, **i32))
    tki_h = host(torch.full((B, N, k), -7, **i32))
    tkv_h = host(torch.full((B, N, k), np.nan, dtype=torch.float32))
    n = _abi.dspark_step_host_workspace_size(cfg, head.struct())
    assert n > 0
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    _abi.check(_abi.dspark_step_host(
        cfg, head.struct(), hidden_h.data_ptr(), anchors_h.data_ptr(), target_h.data_ptr(),
        draft_h.data_ptr(), nd_h.data_ptr(), acc_h.data_ptr(), bon_h.data_ptr(),
        tki_h.data_ptr() if with_topk else 0, tkv_h.data_ptr() if with_topk else 0,
        ws.data_ptr(), n, stream.cuda_stream,
        conf_hidden_h=None if ch_h is None else ch_h.data_ptr()))
    torch.cuda.synchronize()
    assert tio.device_status(ws) == 0

    assert np.array_equal(draft_h.numpy(), g["draft"])
    assert np.array_equal(nd_h.numpy(), g["n_draft"])
    if with_topk:
        assert np.array_equal(tki_h.numpy(), g["topk_ids"])
        assert np.array_equal(tkv_h.numpy(), g["topk_vals"])
    else:
        assert (tki_h.numpy() == -7).all()            # left untouched
    a, b, _ = oracle_verify(g["draft"], g["n_draft"], target)
    assert np.array_equal(acc_h.numpy(), a)
    assert np.array_equal(bon_h.numpy(), b)
