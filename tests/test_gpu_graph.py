"""A pass (dspark_propose + dspark_verify) captured into a CUDA graph and replayed: the
replay equals a direct call, and it reads the live input buffers, so a decoding loop can
refill them and replay the graph each step."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from dspark_block_drafter_gb300 import torch_io as tio  # noqa: E402
from workloads import Workload, make_batch, make_head, make_target  # noqa: E402


def _wl(dtype):
    return Workload("graph_" + dtype, B=32, L_in=8, H=256, V=4096, r=32, top_k=4,
                    sample_from_anchor=True, conf_min=0.5, dtype=dtype, weight_std=0.1,
                    conf_std=0.05, accept_p=0.4, seed=515)


def _outputs(out, acc, bon):
    g = out.numpy()
    g["accepted"] = acc.cpu().numpy()
    g["bonus"] = bon.cpu().numpy()
    return g


@pytest.mark.parametrize("dtype,chain", [("f32", "dense"), ("bf16", "dense"),
                                         ("bf16", "pruned")])
def test_pass_replays_from_a_cuda_graph(dtype, chain):
    wl = _wl(dtype)
    hd = make_head(wl)
    bt, bt2 = make_batch(wl), make_batch(wl, batch_index=1)
    cfg = tio.make_config(wl.B, wl.L_in, wl.H, wl.V, wl.r, wl.top_k, wl.sample_from_anchor,
                          wl.conf_min, wl.dtype, wl.topk_markov)
    head = tio.head_to_device(hd)
    if chain == "pruned":
        head.prepare(cfg)
    hidden = tio.to_device(bt["hidden"])
    anchors = tio.to_device(bt["anchors"])
    out = tio.Outputs.allocate(wl.B, wl.N, wl.top_k, head.V_head)
    ws = tio.workspace_for(cfg, head)
    acc = torch.empty(wl.B, dtype=torch.int32, device="cuda")
    bon = torch.empty_like(acc)
    rng = np.random.default_rng(7)
    target = tio.to_device(rng.integers(0, wl.V, (wl.B, wl.N + 1)).astype(np.int32))

    def one_pass(stream):
        tio.propose(cfg, head, hidden, anchors, out, ws, stream)
        tio.verify(out.draft, out.n_draft, target, acc, bon, None, stream)

    # direct calls first (also the library's one-time per-device set-up)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        one_pass(side)
        one_pass(side)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    direct = _outputs(out, acc, bon)
    assert tio.device_status(ws) == 0

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        one_pass(torch.cuda.current_stream())

    # the replay writes every output afresh
    for t in (out.draft, out.n_draft, acc, bon):
        t.fill_(-7)
    g.replay()
    torch.cuda.synchronize()
    replay = _outputs(out, acc, bon)
    assert tio.device_status(ws) == 0
    for k in direct:
        if direct[k] is not None:
            assert np.array_equal(replay[k], direct[k], equal_nan=True), k

    # new inputs in the same buffers: the replay follows them, as a direct call does
    hidden.copy_(tio.to_device(bt2["hidden"]))
    anchors.copy_(tio.to_device(bt2["anchors"]))
    target.copy_(tio.to_device(make_target(wl, direct["draft"], 1)))
    g.replay()
    torch.cuda.synchronize()
    replay2 = _outputs(out, acc, bon)
    one_pass(torch.cuda.current_stream())
    torch.cuda.synchronize()
    direct2 = _outputs(out, acc, bon)
    assert tio.device_status(ws) == 0
    for k in direct2:
        if direct2[k] is not None:
            assert np.array_equal(replay2[k], direct2[k], equal_nan=True), k
    assert not np.array_equal(direct2["draft"], direct["draft"])
