"""dspark_pass_stats: the counters of the latest propose call on a workspace.

  * loose Cauchy-Schwarz bounds (large Markov weights): the pruned walk evaluates slots
    on the fly, and the counters say how many; a second call on the same workspace
    reports the same counts (they restart with every call), and the results still match
    the oracle;
  * every head row tied (zero lm_head and markov_w2): the dense chain's top-k lists
    overflow for every (slot, block) and are recomputed over every row.
"""
import numpy as np
import pytest

from gpu_cases import compare, oracle_run
from workloads import Workload, make_batch, make_head

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from dspark_block_drafter_gb300 import torch_io as tio  # noqa: E402


def _run(wl, hd, bt, prepare, calls=1):
    cfg = tio.make_config(wl.B, wl.L_in, wl.H, wl.V, wl.r, wl.top_k, wl.sample_from_anchor,
                          wl.conf_min, wl.dtype, wl.topk_markov)
    head = tio.head_to_device(hd)
    if prepare:
        head.prepare(cfg)
    hidden, anchors = tio.to_device(bt["hidden"]), tio.to_device(bt["anchors"])
    out = tio.Outputs.allocate(wl.B, wl.N, wl.top_k, head.V_head)
    ws = tio.workspace_for(cfg, head)
    stats = []
    for _ in range(calls):
        tio.propose(cfg, head, hidden, anchors, out, ws)
        torch.cuda.synchronize()
        assert tio.device_status(ws) == 0
        stats.append(tio.pass_stats(ws))
    return out.numpy(), stats


def test_pruned_walk_counts_slots_evaluated_on_the_fly():
    wl = Workload("loose", B=5, L_in=4, H=64, V=8192, r=64, top_k=8, sample_from_anchor=True,
                  conf_min=0.5, dtype="bf16", weight_std=1.0, conf_std=0.05, seed=77)
    hd, bt = make_head(wl), make_batch(wl)
    g, stats = _run(wl, hd, bt, prepare=True, calls=2)
    st = stats[0]
    assert 0 < st["on_the_fly"] <= wl.B * wl.N
    assert 0 <= st["every_row"] <= st["on_the_fly"]
    assert st["dense_overflow"] == 0
    assert stats[1] == st                       # restarted, not accumulated
    rep = compare(wl, hd, bt, oracle_run(wl, hd, bt), g)
    assert rep["failures"] == [], rep


def test_dense_chain_counts_overflowing_topk_lists():
    wl = Workload("ties", B=3, L_in=5, H=64, V=2048, r=32, top_k=4, sample_from_anchor=True,
                  conf_min=0.0, dtype="bf16", weight_std=0.1, conf_std=0.05, seed=78)
    hd, bt = make_head(wl), make_batch(wl)
    hd["lm_head"] = np.zeros_like(hd["lm_head"])         # z = 0 everywhere
    hd["markov_w2"] = np.zeros_like(hd["markov_w2"])     # and no Markov term: all tied
    g, stats = _run(wl, hd, bt, prepare=False)
    st = stats[0]
    assert st["dense_overflow"] == wl.B * wl.N
    assert st["on_the_fly"] == 0 and st["every_row"] == 0
    # every slot: the lowest rows, in order
    assert np.all(g["draft"] == 0)
    assert np.array_equal(g["topk_ids"], np.broadcast_to(np.arange(wl.top_k), g["topk_ids"].shape))
    rep = compare(wl, hd, bt, oracle_run(wl, hd, bt), g)
    assert rep["failures"] == [], rep
