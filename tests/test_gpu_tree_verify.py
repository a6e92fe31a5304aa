"""dspark_tree_verify on the GPU against the oracle's tree_verify, on identical inputs:
random candidate lattices with targets that follow the lattice for a seeded prefix, and
the lattice of a real proposal at full size."""
import numpy as np
import pytest

from oracle import tree_verify as oracle_tree_verify, verify as oracle_verify
from workloads import WORKLOADS, Workload, make_batch, make_head, make_lattice_target

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from dspark_block_drafter_gb300 import torch_io as tio  # noqa: E402


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()


def _gpu_tree(ids, n_draft, target, outputs=True):
    ids_d, nd_d, t_d = _dev(ids), _dev(n_draft), _dev(target)
    B, N, k = ids_d.shape
    acc = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    bon = torch.full((B,), -9, dtype=torch.int32, device="cuda")
    em = torch.full((B, N + 1), -9, dtype=torch.int32, device="cuda") if outputs else None
    path = torch.full((B, N), -9, dtype=torch.int32, device="cuda") if outputs else None
    tio.tree_verify(ids_d, nd_d, t_d, acc, bon, em, path)
    torch.cuda.synchronize()
    return (acc.cpu().numpy(), bon.cpu().numpy(),
            None if em is None else em.cpu().numpy(),
            None if path is None else path.cpu().numpy())


def _lattice(rng, B, N, k, V):
    return np.array([[rng.choice(V, k, replace=False) for _ in range(N)] for _ in range(B)])


def _same_as_oracle(ids, n_draft, target):
    a, b, e, p = _gpu_tree(ids, n_draft, target)
    a2, b2, e2, p2 = oracle_tree_verify(ids, n_draft, target)
    assert np.array_equal(a, a2) and np.array_equal(b, b2)
    assert np.array_equal(e, e2) and np.array_equal(p, p2)
    return a


@pytest.mark.parametrize("N", [1, 5, 31, 32, 33, 70])
@pytest.mark.parametrize("k", [1, 3, 8, 32])
def test_random_lattices(N, k):
    rng = np.random.default_rng(1000 * N + k)
    B, V = 37, 4000
    wl = Workload("lat", B=B, L_in=N, H=8, V=V, r=1, top_k=k, sample_from_anchor=True,
                  conf_min=0.0, dtype="f32", weight_std=1.0, conf_std=1.0, accept_p=0.15,
                  seed=N * 100 + k)
    ids = _lattice(rng, B, N, k, V)
    target = make_lattice_target(wl, ids)
    n_draft = rng.integers(-2, N + 3, B)            # includes values to clamp
    a = _same_as_oracle(ids, n_draft, target)
    assert a.max() > 0


def test_every_depth_missed_once():
    rng = np.random.default_rng(7)
    N, k, V = 20, 4, 300
    rows = []
    for j in range(N):
        ids = _lattice(rng, 1, N, k, V)[0]
        ranks = rng.integers(0, k, N)
        t = np.array([ids[i, ranks[i]] for i in range(N)] + [5])
        t[j] = next(x for x in range(V) if x not in ids[j])
        rows.append((ids, t))
    ids = np.stack([r[0] for r in rows])
    target = np.stack([r[1] for r in rows])
    for nd in (0, 7, N):
        a = _same_as_oracle(ids, np.full(N, nd), target)
        assert a.tolist() == [min(j, nd) for j in range(N)]


def test_top1_lattice_equals_verify():
    rng = np.random.default_rng(8)
    B, N, V = 64, 16, 50
    ids = rng.integers(0, V, (B, N, 1))
    target = rng.integers(0, V, (B, N + 1))
    agree = rng.integers(0, N + 1, B)
    for b in range(B):
        target[b, :agree[b]] = ids[b, :agree[b], 0]
    n_draft = rng.integers(0, N + 1, B)
    a, b_, e, _ = _gpu_tree(ids, n_draft, target)
    a2, b2, e2 = oracle_verify(ids[:, :, 0], n_draft, target)
    assert np.array_equal(a, a2) and np.array_equal(b_, b2) and np.array_equal(e, e2)


def test_optional_outputs_left_out():
    rng = np.random.default_rng(9)
    ids = _lattice(rng, 9, 6, 3, 40)
    target = rng.integers(0, 40, (9, 7))
    a, b, e, p = _gpu_tree(ids, np.full(9, 6), target, outputs=False)
    a2, b2, _, _ = oracle_tree_verify(ids, np.full(9, 6), target)
    assert np.array_equal(a, a2) and np.array_equal(b, b2)


@pytest.mark.parametrize("name", ["qwen3_8b_b32", "qwen38_27b_b8"])
def test_lattice_of_a_full_size_proposal(name):
    # the GPU's own top-k lattice at the workload's full size (pruned chain, as in the
    # benchmark), verified against targets that follow it for a seeded prefix
    from gpu_cases import gpu_propose
    wl = WORKLOADS[name]
    hd, bt = make_head(wl), make_batch(wl)
    g, _ = gpu_propose(wl, hd, bt, chain="pruned")
    target = make_lattice_target(wl, g["topk_ids"])
    a = _same_as_oracle(g["topk_ids"], g["n_draft"], target)
    assert (a <= g["n_draft"]).all()
