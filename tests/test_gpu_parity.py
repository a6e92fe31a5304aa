"""GPU path (through the C ABI) against the oracle on the same seeded inputs.

Small cases span several tiles and a ragged vocabulary tail; the five named workloads
run at their full sizes.
"""
import numpy as np
import pytest

from workloads import WORKLOADS, Workload, make_batch, make_head

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from gpu_cases import TOL, compare, gpu_propose, oracle_run, run_case  # noqa: E402


def _small(**kw):
    base = dict(name="small", B=3, L_in=5, H=200, V=1000, r=24, top_k=5,
                sample_from_anchor=True, conf_min=0.5, dtype="bf16", weight_std=0.2,
                conf_std=0.05, seed=4242)
    base.update(kw)
    return Workload(**base)


def test_tiny_fp32_workload():
    g, o, rep = run_case(WORKLOADS["tiny_fp32"])
    assert rep["slots"] == 8


CHAINS = ["dense", "pruned"]


@pytest.mark.parametrize("shape", [
    dict(B=6, L_in=5),                                  # 30 prediction rows: tiled GEMM,
                                                        # chain in one chunk of 6 blocks
    dict(B=10, L_in=3, top_k=3),                        # two chunks of blocks
    dict(B=3, L_in=5, r=48),                            # rank above the register cache
    dict(B=2, L_in=4, H=1200),                          # 8 rows, hidden past 32 KB: the
                                                        # few-row GEMM, chain alone
    dict(B=2, L_in=4, H=64, V=40960, r=16, top_k=8),    # more rows than threads x CTAs:
                                                        # several rows per thread
    dict(B=3, L_in=6, sample_from_anchor=False, topk_markov=False),
])
def test_fp32_chain_shapes(shape):
    # the fp32 path's launch forms: one launch (small problems) or GEMM + chain, blocks in
    # chunks, the markov_w2 column in registers or streamed, one or several rows a thread
    run_case(_small(dtype="f32", **shape))


@pytest.mark.parametrize("sfa", [True, False])
@pytest.mark.parametrize("topk_markov", [True, False])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_small_dense(sfa, topk_markov, dtype):
    run_case(_small(sample_from_anchor=sfa, topk_markov=topk_markov, dtype=dtype))


@pytest.mark.parametrize("sfa", [True, False])
@pytest.mark.parametrize("topk_markov", [True, False])
@pytest.mark.parametrize("k", [1, 5, 32])
def test_small_pruned(sfa, topk_markov, k):
    run_case(_small(sample_from_anchor=sfa, topk_markov=topk_markov, top_k=k), chain="pruned")


@pytest.mark.parametrize("shape", [
    dict(B=4, L_in=8),                                  # 32 prediction rows per tile
    dict(B=2, L_in=16, V=1000),                         # ragged vocabulary tail
    dict(B=16, L_in=3, sample_from_anchor=False),       # 1+N layout, 2 slots
    dict(B=32, L_in=16, H=520, V=777 * 8),              # ragged K, several tiles
])
@pytest.mark.parametrize("chain", CHAINS)
def test_even_slot_shapes(shape, chain):
    # whole-block tiles of 32 prediction rows, ragged vocabulary and K tails
    run_case(_small(**shape), chain=chain)


@pytest.mark.parametrize("chain", CHAINS)
def test_pruned_loose_bounds_many_candidates(chain):
    # large Markov weights: the Cauchy-Schwarz bounds admit most rows, so the pruned
    # chain has to evaluate and reduce its candidate buffer many times
    wl = _small(B=5, L_in=4, H=64, V=8192, r=64, top_k=8, weight_std=1.0, seed=77)
    run_case(wl, chain=chain)


@pytest.mark.parametrize("chain", CHAINS)
@pytest.mark.parametrize("form", ["full", "d2t"])
@pytest.mark.parametrize("sfa", [True, False])
def test_small_reduced_vocab(form, sfa, chain):
    wl = _small(n_emit=304, sample_from_anchor=sfa, V=1024)
    g, o, rep = run_case(wl, form, chain=chain)
    emit = set(make_head(wl)["emit_rows"].tolist())
    assert set(g["draft"].ravel().tolist()) <= emit
    assert set(g["topk_ids"].ravel().tolist()) <= emit


@pytest.mark.parametrize("chain", CHAINS)
def test_single_block_single_slot(chain):
    run_case(_small(B=1, L_in=1, top_k=3), chain=chain)


@pytest.mark.parametrize("chain", CHAINS)
def test_topk_equals_head_rows(chain):
    # k = V_head: every row is a candidate; ragged tiny vocabulary
    wl = _small(V=1000, n_emit=32, top_k=32, L_in=3)
    run_case(wl, "d2t", chain=chain)


@pytest.mark.parametrize("chain", CHAINS)
def test_large_rank_and_many_blocks(chain):
    run_case(_small(B=40, L_in=3, r=300, H=136, V=520, top_k=2), chain=chain)


def test_anchor_is_last_token():
    wl = _small()
    hd, bt = make_head(wl), make_batch(wl)
    bt["anchors"][:] = wl.V - 1
    run_case(wl, hd=hd, bt=bt)


def test_confidence_at_threshold_keeps_slot():
    # w_conf = 0, b_conf = 0 gives conf = 0.5 exactly on both sides
    wl = _small(conf_min=0.5)
    hd, bt = make_head(wl), make_batch(wl)
    hd["w_conf"] = np.zeros_like(hd["w_conf"])
    g, o, rep = run_case(wl, hd=hd, bt=bt)
    assert np.all(g["conf"] == 0.5)
    assert np.all(g["n_draft"] == wl.N)


def test_truncation_everywhere():
    # strong confidence head: truncation lands on many different slots
    wl = _small(B=24, L_in=8, conf_std=0.3, conf_min=0.5)
    g, o, rep = run_case(wl)
    assert len(set(g["n_draft"].tolist())) > 2


def test_zero_markov_is_plain_argmax():
    wl = _small()
    hd, bt = make_head(wl), make_batch(wl)
    hd["markov_w1"] = np.zeros_like(hd["markov_w1"])
    g, o, rep = run_case(wl, hd=hd, bt=bt)


def test_bad_anchor_sets_device_status():
    import dspark_block_drafter_gb300 as ds
    from dspark_block_drafter_gb300 import torch_io as tio
    wl = _small()
    hd, bt = make_head(wl), make_batch(wl)
    bt["anchors"][1] = wl.V + 5
    cfg = tio.make_config(wl.B, wl.L_in, wl.H, wl.V, wl.r, wl.top_k, True, wl.conf_min, "bf16")
    head = tio.head_to_device(hd)
    out = tio.Outputs.allocate(wl.B, wl.N, wl.top_k, wl.V)
    ws = tio.workspace_for(cfg, head)
    tio.propose(cfg, head, tio.to_device(bt["hidden"]), tio.to_device(bt["anchors"]), out, ws)
    assert tio.device_status(ws) == ds._abi.DSPARK_ERR_DEVICE
    assert tio.device_status(ws) == 0          # the word is cleared once read


def test_repeat_calls_same_workspace_identical():
    wl = _small()
    hd, bt = make_head(wl), make_batch(wl)
    g1, ws = gpu_propose(wl, hd, bt)
    g2, _ = gpu_propose(wl, hd, bt)
    for k in ("draft", "topk_ids", "n_draft"):
        assert np.array_equal(g1[k], g2[k])
    assert np.array_equal(g1["topk_vals"], g2["topk_vals"])


# ------------------------------------------------------------------ full sizes
@pytest.mark.parametrize("name", ["qwen3_8b_b1", "qwen3_8b_b32", "qwen38_27b_b8",
                                  "gemma4_bonus_b64"])
def test_full_size_workload(name):
    wl = WORKLOADS[name]
    hd, bt = make_head(wl), make_batch(wl)
    forms = ["full", "d2t"] if wl.n_emit else ["full"]
    o = oracle_run(wl, hd, bt)
    for form in forms:
        for chain in CHAINS:
            g, _ = gpu_propose(wl, hd, bt, form, chain=chain)
            rep = compare(wl, hd, bt, o, g, form)
            assert rep["failures"] == [], (form, chain, rep)


# ------------------------------------------------------------------ plan and limit edges
@pytest.mark.parametrize("H", [192, 320])
@pytest.mark.parametrize("chain", CHAINS)
def test_ragged_last_k_stage(H, chain):
    # H/64 odd: stages of two K-blocks end with one whose second half lies past H
    run_case(_small(B=32, L_in=8, H=H, V=2048), chain=chain)


@pytest.mark.parametrize("chain", CHAINS)
def test_blocks_beyond_one_tile(chain):
    # more than 256 blocks: several block tiles, the last one ragged
    run_case(_small(B=300, L_in=2, H=64, V=512, r=16, top_k=2), chain=chain)


@pytest.mark.parametrize("chain", CHAINS)
def test_bonus_layout_six_slots(chain):
    # the 1+N layout with 6 prediction slots and 64 blocks (32-block tiles of 6 slots)
    run_case(_small(B=64, L_in=7, sample_from_anchor=False, H=128, V=1024, r=32, top_k=1),
             chain=chain)


@pytest.mark.parametrize("shape", [
    # several pair tiles, ragged vocabulary tail, an odd number of K-blocks
    dict(B=64, L_in=7, sample_from_anchor=False, H=576, V=3000, r=32, top_k=4),
    # fewer blocks than the tile holds (the hidden box reads zeros past them)
    dict(B=48, L_in=7, sample_from_anchor=False, H=256, V=2048, r=32, top_k=1),
    dict(B=40, L_in=6, H=320, V=1504, r=24, top_k=8),
])
@pytest.mark.parametrize("chain", CHAINS)
def test_six_slot_block_tiles(shape, chain):
    # six slots of 33-64 blocks: pair tiles over two block tiles of 32, the second
    # partly empty when B < 64
    run_case(_small(**shape), chain=chain)


@pytest.mark.parametrize("chain", CHAINS)
@pytest.mark.parametrize("form", ["full", "d2t"])
def test_six_slot_reduced_vocab(form, chain):
    wl = _small(B=64, L_in=7, sample_from_anchor=False, H=192, V=4096, r=32, top_k=2,
                n_emit=1000)
    g, o, rep = run_case(wl, form, chain=chain)
    emit = set(make_head(wl)["emit_rows"].tolist())
    assert set(g["draft"].ravel().tolist()) <= emit


@pytest.mark.parametrize("shape", [
    # two N-tiles of 256 prediction rows (B=32 x 16 slots); H = 320: five K-blocks in
    # three stages, the last one half past H
    dict(B=32, L_in=16, H=320, V=152 * 256 + 200, r=24, top_k=8),
    # one N-tile (B=32 x 8 slots), ragged vocabulary tail
    dict(B=32, L_in=8, H=320, V=160 * 256 + 64, r=24, top_k=4),
    # six slots of 64 blocks
    dict(B=64, L_in=7, sample_from_anchor=False, H=256, V=80 * 256, r=32, top_k=1),
])
@pytest.mark.parametrize("chain", CHAINS)
def test_several_tile_waves(shape, chain):
    # more 256-row pair tiles than pairs (76 on 152 SMs), not a whole number of waves
    run_case(_small(**shape), chain=chain)


@pytest.mark.parametrize("chain", CHAINS)
def test_most_slots(chain):
    # 256 prediction slots: the longest chain the bf16 path takes
    run_case(_small(B=2, L_in=256, H=64, V=512, r=16, top_k=3), chain=chain)


@pytest.mark.parametrize("chain", CHAINS)
def test_largest_rank(chain):
    # Markov rank 512: the largest the bf16 path takes
    run_case(_small(B=8, L_in=4, H=64, V=512, r=512, top_k=4), chain=chain)


def test_bad_anchor_sets_device_status_pruned():
    import dspark_block_drafter_gb300 as ds
    from dspark_block_drafter_gb300 import torch_io as tio
    wl = _small(r=32)
    hd, bt = make_head(wl), make_batch(wl)
    bt["anchors"][2] = -3
    cfg = tio.make_config(wl.B, wl.L_in, wl.H, wl.V, wl.r, wl.top_k, True, wl.conf_min, "bf16")
    head = tio.head_to_device(hd).prepare(cfg)
    out = tio.Outputs.allocate(wl.B, wl.N, wl.top_k, wl.V)
    ws = tio.workspace_for(cfg, head)
    tio.propose(cfg, head, tio.to_device(bt["hidden"]), tio.to_device(bt["anchors"]), out, ws)
    assert tio.device_status(ws) == ds._abi.DSPARK_ERR_DEVICE
    assert tio.device_status(ws) == 0


# ------------------------------------------------------------------ pair tiles of exactly
# 256 prediction rows, which the lm_head GEMM runs with the prediction rows on the MMA's M
@pytest.mark.parametrize("H", [256, 200, 320])
def test_pm_tiles_h_stages(H):
    # H = 256: two K-blocks per stage; 200: one per stage; 320: a ragged last stage
    run_case(_small(B=32, L_in=8, H=H, V=1000, r=16, top_k=3), chain="pruned")


def test_pm_tiles_ragged_slots_and_blocks():
    # 15 slots in chunks of 8 and 7; 70 blocks in tiles of 64 and 6
    run_case(_small(B=32, L_in=15, H=128, V=2048, r=16, top_k=2), chain="pruned")
    run_case(_small(B=70, L_in=4, H=128, V=1024, r=16, top_k=2), chain="pruned")


@pytest.mark.parametrize("form", ["full", "d2t"])
@pytest.mark.parametrize("sfa", [True, False])
def test_pm_tiles_reduced_vocab(form, sfa):
    wl = _small(B=32, L_in=9 if not sfa else 8, H=128, n_emit=304, sample_from_anchor=sfa, V=1024)
    g, o, rep = run_case(wl, form, chain="pruned")
    emit = set(make_head(wl)["emit_rows"].tolist())
    assert set(g["draft"].ravel().tolist()) <= emit


# ------------------------------------------------------------------ z tiles left out by the
# GEMM (pair tiles of 256 prediction rows, top-k over corrected logits)
@pytest.mark.parametrize("weight_std", [0.05, 1.0])
def test_pm_skip_markov_scale(weight_std):
    # a small Markov term leaves most tiles out; a large one keeps most of them
    run_case(_small(B=32, L_in=8, H=128, V=4096, r=32, top_k=4, weight_std=weight_std,
                    seed=911), chain="pruned")


def test_pm_skip_without_topk_outputs():
    # no top-k asked: the bound is of rank 1
    from gpu_cases import gpu_propose, oracle_run, compare
    wl = _small(B=32, L_in=8, H=128, V=4096, r=32, top_k=4, seed=912)
    hd, bt = make_head(wl), make_batch(wl)
    g, _ = gpu_propose(wl, hd, bt, want_topk=False, chain="pruned")
    rep = compare(wl, hd, bt, oracle_run(wl, hd, bt), g)
    assert rep["failures"] == [], rep


def test_pm_no_skip_for_base_logit_topk():
    # top-k of the base logits: every tile is stored
    run_case(_small(B=32, L_in=8, H=128, V=2048, r=32, top_k=6, topk_markov=False),
             chain="pruned")


def test_pm_skip_with_every_row_fallback():
    # Zero hidden states and a +4 bias on the first 640 of 4096 rows: every hot row ties on
    # z, so the candidate lists overflow and each slot is evaluated over every row, while
    # the 27 cold tiles sit far below the threshold and are left out of z.
    wl = _small(B=32, L_in=8, H=128, V=4096, r=32, top_k=4, seed=913)
    hd, bt = make_head(wl), make_batch(wl)
    bt["hidden"] = np.zeros_like(bt["hidden"])
    bias = np.zeros(wl.V, np.float32)
    bias[:640] = 4.0
    hd["lm_bias"] = bias
    g, o, rep = run_case(wl, hd=hd, bt=bt, chain="pruned")
    assert (g["draft"] < 640).all()


# ------------------------------------------------------------------ slot counts that do not
# fill 256-row tiles (7 and 6 slots; one, two and three block tiles)
@pytest.mark.parametrize("B,L_in,sfa", [(32, 7, True), (64, 7, False), (96, 7, False)])
def test_odd_slot_counts_pruned(B, L_in, sfa):
    run_case(_small(B=B, L_in=L_in, sample_from_anchor=sfa, H=128, V=2048, r=16, top_k=3),
             chain="pruned")


# ------------------------------------------------------------------ a prepared buffer used
# with another head: nothing past its header is read, the error word says why
@pytest.mark.parametrize("change", ["markov_w2 address", "rank", "head rows"])
def test_prepared_buffer_for_another_head(change):
    import dspark_block_drafter_gb300 as ds
    from dspark_block_drafter_gb300 import torch_io as tio
    wl = _small(r=32, V=1024, B=32, L_in=8, H=256, weight_std=0.1)
    hd, bt = make_head(wl), make_batch(wl)
    cfg = tio.make_config(wl.B, wl.L_in, wl.H, wl.V, wl.r, wl.top_k, True, wl.conf_min, "bf16")
    head = tio.head_to_device(hd).prepare(cfg)
    hidden, anchors = tio.to_device(bt["hidden"]), tio.to_device(bt["anchors"])
    if change == "markov_w2 address":            # same sizes, other weights
        other = head.markov_w2.clone()
        use_cfg, use = cfg, tio.Head(head.lm_head, head.markov_w1, other, None, None,
                                     head.w_conf, head.b_conf, head.prepared)
    elif change == "rank":                       # prepared for r = 32, used with r = 16
        wl2 = _small(r=16, V=1024, B=32, L_in=8, H=256, weight_std=0.1)
        hd2 = make_head(wl2)
        use_cfg = tio.make_config(wl.B, wl.L_in, wl.H, wl.V, 16, wl.top_k, True,
                                  wl.conf_min, "bf16")
        h2 = tio.head_to_device(hd2)
        use = tio.Head(h2.lm_head, h2.markov_w1, h2.markov_w2, None, None, h2.w_conf,
                       h2.b_conf, head.prepared)
    else:                                        # the compact form of fewer head rows
        rows = np.sort(np.random.default_rng(3).choice(wl.V, 512, replace=False))
        hd["emit_rows"] = rows
        hd["lm_bias"] = np.zeros(wl.V, np.float32)
        h2 = tio.head_to_device(hd, "d2t")
        use_cfg, use = cfg, tio.Head(h2.lm_head, h2.markov_w1, h2.markov_w2, h2.lm_bias,
                                     h2.d2t, h2.w_conf, h2.b_conf, head.prepared)
    out = tio.Outputs.allocate(wl.B, wl.N, wl.top_k, use.V_head)
    ws = tio.workspace_for(use_cfg, use)
    tio.propose(use_cfg, use, hidden, anchors, out, ws)
    assert tio.device_status(ws) == ds._abi.DSPARK_ERR_DEVICE
    assert "prepared" in ds._abi.dspark_last_error()
    assert tio.device_status(ws) == 0
    # the same workspace, with a buffer prepared for this head, is clean again
    use.prepare(use_cfg)
    tio.propose(use_cfg, use, hidden, anchors, out, ws)
    assert tio.device_status(ws) == 0


# ------------------------------------------------------------------ a separate confidence
# input: the confidence head reads it, the logits and the chain do not
@pytest.mark.parametrize("chain,sfa,dtype", [("dense", True, "bf16"), ("pruned", False, "bf16"),
                                             ("pruned", True, "bf16"), ("dense", True, "f32")])
def test_separate_confidence_input(chain, sfa, dtype):
    from workloads import make_conf_hidden
    wl = _small(sample_from_anchor=sfa, dtype=dtype, r=32, conf_std=0.3, L_in=7)
    hd, bt = make_head(wl), make_batch(wl)
    ch = make_conf_hidden(wl)
    g, o, rep = run_case(wl, chain=chain, hd=hd, bt=bt, conf_hidden=ch)
    plain, _ = gpu_propose(wl, hd, bt, chain=chain)
    for key in ("draft", "topk_ids"):
        assert np.array_equal(g[key], plain[key]), key
    assert not np.allclose(g["conf"], plain["conf"])
    # the hidden states themselves as the separate input change nothing
    same, _ = gpu_propose(wl, hd, bt, chain=chain, conf_hidden=bt["hidden"])
    for key in ("draft", "topk_ids", "topk_vals", "conf", "n_draft"):
        assert np.array_equal(same[key], plain[key]), key


def test_separate_confidence_input_full_size():
    from workloads import make_conf_hidden
    wl = WORKLOADS["qwen3_8b_b32"]
    hd, bt = make_head(wl), make_batch(wl)
    run_case(wl, chain="pruned", hd=hd, bt=bt, conf_hidden=make_conf_hidden(wl))


def test_separate_confidence_input_adaptive():
    from workloads import make_conf_hidden
    wl = _small(r=32, conf_std=0.3, L_in=9, B=5)
    hd, bt = make_head(wl), make_batch(wl)
    run_case(wl, chain="pruned", hd=hd, bt=bt, conf_hidden=make_conf_hidden(wl),
             skip_truncated=True)
