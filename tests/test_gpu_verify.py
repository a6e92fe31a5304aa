"""dspark_verify on the GPU against the oracle's verify, on identical inputs."""
import numpy as np
import pytest

from oracle import check, propose as oracle_propose, verify as oracle_verify
from workloads import WORKLOADS, make_batch, make_head, make_target

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from dspark_block_drafter_gb300 import torch_io as tio  # noqa: E402


def _gpu_verify(draft, n_draft, target, with_emitted=True):
    d = torch.from_numpy(np.ascontiguousarray(draft, np.int32)).cuda()
    n = torch.from_numpy(np.ascontiguousarray(n_draft, np.int32)).cuda()
    t = torch.from_numpy(np.ascontiguousarray(target, np.int32)).cuda()
    B, N = d.shape
    acc = torch.empty(B, dtype=torch.int32, device="cuda")
    bon = torch.empty(B, dtype=torch.int32, device="cuda")
    em = torch.empty(B, N + 1, dtype=torch.int32, device="cuda") if with_emitted else None
    tio.verify(d, n, t, acc, bon, em)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), bon.cpu().numpy(), None if em is None else em.cpu().numpy()


def test_tiny_workload_oracle_draft():
    wl = WORKLOADS["tiny_fp32"]
    hd, bt = make_head(wl), make_batch(wl)
    o = oracle_propose(bt["hidden"], bt["anchors"], hd["lm_head"], hd["markov_w1"],
                       hd["markov_w2"], L_in=wl.L_in, sample_from_anchor=True,
                       top_k=wl.top_k, conf_min=wl.conf_min, w_conf=hd["w_conf"])
    target = make_target(wl, o["draft"])
    a, b, e = _gpu_verify(o["draft"], o["n_draft"], target)
    assert check.check_verify(o["draft"], o["n_draft"], target, a, b, e) == []
    assert np.all(a < wl.N)         # one planted mismatch per block


@pytest.mark.parametrize("N", [1, 6, 16, 31, 32, 33, 70])
def test_planted_mismatch_every_position(N):
    rng = np.random.default_rng(N)
    V = 5000
    rows = []
    for nd in sorted({0, 1, N // 2, N}):
        for j in range(N):
            d = rng.integers(0, V, N)
            t = np.concatenate([d, rng.integers(0, V, 1)])
            t[j] = (d[j] + 1 + rng.integers(0, V - 1)) % V
            rows.append((d, nd, t))
        d = rng.integers(0, V, N)                    # all agree
        rows.append((d, nd, np.concatenate([d, rng.integers(0, V, 1)])))
    draft = np.stack([r[0] for r in rows])
    n_draft = np.array([r[1] for r in rows])
    target = np.stack([r[2] for r in rows])
    a, b, e = _gpu_verify(draft, n_draft, target)
    assert check.check_verify(draft, n_draft, target, a, b, e) == []
    # greedy lossless: what is emitted is the target's own prefix
    for i in range(len(rows)):
        assert e[i, :a[i] + 1].tolist() == target[i, :a[i] + 1].tolist()


def test_ndraft_clamped_and_no_emitted():
    rng = np.random.default_rng(3)
    draft = rng.integers(0, 10, (4, 5))
    target = np.concatenate([draft, rng.integers(0, 10, (4, 1))], axis=1)
    n = np.array([-3, 0, 5, 99])
    a, b, _ = _gpu_verify(draft, n, target, with_emitted=False)
    assert a.tolist() == [0, 0, 5, 5]
    a2, b2, _ = oracle_verify(draft, n, target)
    assert a.tolist() == a2.tolist() and b.tolist() == b2.tolist()


@pytest.mark.parametrize("name", ["qwen3_8b_b32", "gemma4_bonus_b64"])
def test_workload_targets(name):
    # drafts of the oracle's shape; agreement prefix from the workload's recipe
    wl = WORKLOADS[name]
    rng = np.random.default_rng(9)
    draft = rng.integers(0, wl.V, (wl.B, wl.N))
    n_draft = rng.integers(0, wl.N + 1, wl.B)
    target = make_target(wl, draft)
    a, b, e = _gpu_verify(draft, n_draft, target)
    assert check.check_verify(draft, n_draft, target, a, b, e) == []


def test_propose_then_verify_properties():
    # the pipeline on the GPU alone: properties that hold for any draft
    from gpu_cases import gpu_propose
    from workloads import Workload
    wl = Workload("pipe", B=16, L_in=6, H=128, V=800, r=16, top_k=2, sample_from_anchor=True,
                  conf_min=0.5, dtype="bf16", weight_std=0.2, conf_std=0.1, accept_p=0.3,
                  seed=5)
    hd, bt = make_head(wl), make_batch(wl)
    g, _ = gpu_propose(wl, hd, bt)
    rng = np.random.default_rng(1)
    target = rng.integers(0, wl.V, (wl.B, wl.N + 1))
    agree = rng.integers(0, wl.N + 1, wl.B)
    for bb in range(wl.B):
        target[bb, :agree[bb]] = g["draft"][bb, :agree[bb]]
    a, b, e = _gpu_verify(g["draft"], g["n_draft"], target)
    for bb in range(wl.B):
        d, t, n = g["draft"][bb], target[bb], g["n_draft"][bb]
        assert 0 <= a[bb] <= n
        assert list(d[:a[bb]]) == list(t[:a[bb]])            # an agreeing prefix ...
        assert a[bb] == n or d[a[bb]] != t[a[bb]]             # ... that is the longest
        assert b[bb] == t[a[bb]]
        assert list(e[bb, :a[bb] + 1]) == list(t[:a[bb] + 1])
