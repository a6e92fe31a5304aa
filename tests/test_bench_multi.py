"""The benchmark's multi-process host logic on the CPU: two `gloo` ranks.

Blocks are independent, so under torchrun every rank runs its own replica and nothing
crosses ranks on the data path.  What the ranks do share is host logic: the step time is
the slowest rank's, the throughput counts every rank's slots, and the reference arm
runs on rank 0 alone.  These tests run that logic with world_size 2 over gloo.
"""
import contextlib
import io
import json
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _throughput_worker(rank, world, port, results):
    _init(rank, world, port)
    try:
        ms = [1.0, 2.5][rank]           # rank 1 is the slow one
        slots = [512, 512][rank]
        results[rank] = bench.job_throughput(ms, slots, world)
    finally:
        dist.destroy_process_group()


def _reference_worker(rank, world, port, results):
    _init(rank, world, port)
    try:
        buf = io.StringIO()
        with contextlib.redirect_stdout(buf):
            rc = bench.main(["--impl", "reference", "--workload", "tiny_fp32", "--steps", "1",
                             "--warmup", "3", "--gpus", str(world)])
        results[rank] = (rc, buf.getvalue())
    finally:
        dist.destroy_process_group()


def _spawn(fn, world=2):
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(fn, args=(world, port, results), nprocs=world, join=True)
        return dict(results)


def test_job_throughput_takes_slowest_rank_and_all_slots():
    res = _spawn(_throughput_worker)
    for rank in (0, 1):
        ms, value = res[rank]
        assert ms == 2.5                                 # the slowest rank's step
        assert value == pytest.approx(1024 / 2.5e-3)     # both ranks' slots


def test_job_throughput_single_process_needs_no_group():
    assert bench.job_throughput(2.0, 512, 1) == (2.0, 512 / 2e-3)


def test_reference_arm_runs_on_rank0_only():
    res = _spawn(_reference_worker)
    rc0, out0 = res[0]
    rc1, out1 = res[1]
    assert rc0 == 0 and rc1 == 0
    assert out1 == ""                                     # the other rank does no work
    lines = [json.loads(x) for x in out0.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["unit"] == "slots/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_parse_clocks_reports_median_and_reasons():
    rows = [
        "2026/01/02 10:00:00.100, 0, 1900, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/01/02 10:00:00.120, 0, 2000, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active",
        "2026/01/02 10:00:00.140, 0, 1950, 2070, 1350.0, 0x4, Not Active, Not Active, Not Active, Active",
        "garbage line",
    ]
    c = bench.parse_clocks(rows)
    assert c == {"sm_mhz": 1950, "sm_max_mhz": 2070, "samples": 3, "window": "whole run",
                 "reasons": ["sw_power_cap"]}
    assert bench.parse_clocks([]) is None


def test_parse_clocks_keeps_the_timed_window():
    import datetime as dt
    rows = [
        "2026/01/02 10:00:00.000, 0, 1000, 2070, 100.0, 0x0, Active, Not Active, Not Active, Not Active",
        "2026/01/02 10:00:00.500, 0, 2010, 2070, 1300.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/01/02 10:00:00.520, 0, 2030, 2070, 1300.0, 0x0, Not Active, Not Active, Not Active, Not Active",
        "2026/01/02 10:00:01.500, 0, 1200, 2070, 300.0, 0x0, Not Active, Active, Not Active, Not Active",
    ]
    t = dt.datetime(2026, 1, 2, 10, 0, 0)
    c = bench.parse_clocks(rows, (t + dt.timedelta(seconds=0.4), t + dt.timedelta(seconds=0.6)))
    # the idle sample before and the slowed one after the window do not count
    assert c == {"sm_mhz": 2020, "sm_max_mhz": 2070, "samples": 2, "window": "timed region",
                 "reasons": []}
    c = bench.parse_clocks(rows, (t + dt.timedelta(seconds=5), t + dt.timedelta(seconds=6)))
    assert c["samples"] == 4 and c["window"].startswith("whole run")


def test_cpu_baseline_sample_within_the_batch():
    from workloads import WORKLOADS, make_batch, make_head
    wl = WORKLOADS["tiny_fp32"]                        # a batch of 2 blocks
    c = bench.cpu_baseline(wl, make_head(wl), make_batch(wl), budget_s=2.0, min_work_s=0.3)
    assert c["sample"].startswith("2 of 2 blocks")
    assert c["kind"] == "oracle" and c["cores"] >= 1 and c["value"] > 0


def test_verify_only_timing_arithmetic(monkeypatch):
    import types

    import torch

    class Event:                       # 2 ms between the two records
        def __init__(self, enable_timing=True):
            pass

        def record(self, stream=None):
            pass

        def elapsed_time(self, other):
            return 2.0

    monkeypatch.setattr(torch.cuda, "Event", Event)
    monkeypatch.setattr(torch.cuda, "synchronize", lambda *a, **k: None)
    calls = []
    tio = types.SimpleNamespace(verify=lambda *a: calls.append(a))
    out = types.SimpleNamespace(draft="d", n_draft="n")
    r = bench._verify_only(tio, out, "t", "a", "b", None, None, K=10, W=3, B=32)
    assert len(calls) == 13 and calls[0][:2] == ("d", "n")
    assert r == {"us_per_call": 200.0, "blocks_per_s": 32 / 200e-6, "calls": 10}

    def broken(*a):
        raise RuntimeError("no device")
    r = bench._verify_only(types.SimpleNamespace(verify=broken), out, "t", "a", "b", None,
                           None, K=10, W=3, B=32)
    assert r == {"unavailable": "RuntimeError: no device"}


@pytest.mark.parametrize("name,v_head,mbytes,gflops", [
    ("qwen3_8b_b1", 151936, 1322.6, 21.2),
    ("qwen3_8b_b32", 151936, 1327.0, 677.1),
    ("qwen38_27b_b8", 248320, 2671.3, 341.8),
    ("gemma4_bonus_b64", 32768, 196.3, 74.1),    # the 32768 emittable rows only
])
def test_algorithmic_work_per_pass(name, v_head, mbytes, gflops):
    # the roofline's numerator: bytes and flops the method must touch per pass, against
    # figures worked out separately from the same definition (lm_head rows needed, the
    # markov_w2 columns needed, gathered markov_w1 rows, hidden, w_conf, outputs and
    # verify I/O; 2·M·H·V_e + 2·M·r·V_e + 2·M·H flops)
    from workloads import WORKLOADS
    a = bench._algorithmic(WORKLOADS[name], v_head)
    assert a["bytes"] / 1e6 == pytest.approx(mbytes, rel=5e-3)
    assert a["flops"] / 1e9 == pytest.approx(gflops, rel=5e-3)
    assert a["gemm_flops"] == 2.0 * WORKLOADS[name].M * WORKLOADS[name].H * v_head
