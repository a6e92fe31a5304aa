#!/usr/bin/env python3
"""Benchmark: DSpark proposal head + greedy verify on one GB300 per process.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

One step is one full pass of the path over one batch: dspark_propose (confidence,
base logits, Markov-corrected greedy chain, top-k, truncation) then dspark_verify.
The default workload is the Qwen3-8B-shaped head at B=32 blocks of L=16 slots
(H=4096, V=151936, r=256, top_k=8, conf_min=0.5).  Inputs are seeded and synthetic.

Timing: W untimed warm-up steps, then K timed steps.  Before every timed step a 512 MB
buffer is written and another 512 MB read (L2 flush, untimed: the read makes the
write's dirty lines go back to HBM before the step); each step is bracketed by CUDA events on the
launching stream, and the library records stage events inside dspark_propose_timed so
the lm_head GEMM's own duration is known.  Under torchrun each rank runs an
independent replica on its own batch (no collective on the data path: blocks are
independent); the step time is the maximum over ranks and ``value`` counts the slots
of all ranks.

``--impl reference`` times the CPU oracle (float64 NumPy) on the host cores on a
bounded sample of the same workload and prints the same JSON line with
"impl": "reference".
"""
from __future__ import annotations

import argparse
import dataclasses
import datetime
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

def metric_of(wl) -> str:
    """The headline metric's name for this workload (the default one: B=32, V=151936)."""
    return f"drafted slots/sec (propose+verify) at B={wl.B}, V={wl.V}"
UNIT = "slots/s"
FLUSH_BYTES = 512 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# DRAM bytes (read + written) of one lm_head GEMM launch from an ncu capture of the
# current kernel, per workload; the summary and the command are in the named file.
GEMM_TRAFFIC = {
    "qwen3_8b_b32": (1.2496e9 + 0.0245e9, "profiles/logits_gemm_qwen3_8b_b32.md"),
    "qwen3_8b_b1": (1.2449e9 + 0.0042e9, "profiles/logits_gemm_qwen3_8b_b1.md"),
    "qwen38_27b_b8": (2.5444e9 + 0.0754e9, "profiles/logits_gemm_qwen38_27b_b8.md"),
    "gemma4_bonus_b64": (0.1870e9 + 0.0071e9, "profiles/logits_gemm_gemma4_bonus_b64.md"),
}
# fp32 CUDA-core peak used for the fp32 path: 152 SMs x 128 FP32 lanes x 2 flops (FMA) x
# 2.07 GHz maximum SM clock
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


class L2Flush:
    """Evicts the step's inputs from L2 between timed steps (untimed): a buffer larger
    than L2 is written, then a second one read, so that the write's dirty lines go back
    to HBM before the step instead of during it."""

    def __init__(self, nbytes, dev):
        import torch
        self.w = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(nbytes // 4, dtype=torch.int32, device=dev)

    def zero_(self):
        self.w.zero_()
        self.r.max()


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["_source"] = "measured"
        return d
    d = dict(FALLBACK_PEAKS)
    d["_source"] = "fallback"
    return d


def _algorithmic(wl, V_head):
    """Algorithmic bytes and flops of one pass (all steps), and of the lm_head GEMM."""
    es = 2 if wl.dtype == "bf16" else 4
    M, H, r, B, N, k = wl.M, wl.H, wl.r, wl.B, wl.N, wl.top_k
    gemm_bytes = V_head * H * es + M * H * es          # lm_head + hidden
    gemm_flops = 2.0 * M * H * V_head
    markov_flops = 2.0 * M * r * V_head
    bytes_all = (V_head * H * es + r * V_head * es + M * r * es + B * wl.L_in * H * es
                 + H * es + (V_head * 4 if wl.n_emit else 0)
                 + B * N * (4 + 4 + 8 * k) + B * (N + 1) * 4 + B * 16)
    flops_all = gemm_flops + markov_flops + 2.0 * M * H
    return dict(gemm_bytes=gemm_bytes, gemm_flops=gemm_flops, bytes=bytes_all,
                flops=flops_all)


class ClockSampler:
    """nvidia-smi clock / throttle samples, every 20 ms, kept for the timed region."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        # raw samples; DSPARK_CLOCKS_DIR keeps them where the caller wants them
        out_dir = os.environ.get("DSPARK_CLOCKS_DIR", tempfile.gettempdir())
        self.path = os.path.join(out_dir, f"dspark_clocks_rank{index}.csv")

    def start(self, ready_timeout_s: float = 5.0):
        """Starts the sampler and returns once its first sample is written (or after
        ready_timeout_s), so that it is live before the timed region begins."""
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-i", str(self.index), "-lms", "20"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < ready_timeout_s and self.proc.poll() is None:
            if os.path.getsize(self.path) > 0:
                break
            time.sleep(0.01)

    def stop(self, window=None):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        with open(self.path) as f:
            return parse_clocks(f, window)


BAD_CLOCK_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def _sample_time(stamp: str):
    try:
        return datetime.datetime.strptime(stamp, "%Y/%m/%d %H:%M:%S.%f")
    except ValueError:
        return None


def parse_clocks(lines, window=None):
    """Summary of nvidia-smi samples (the query columns of ClockSampler.Q, no header):
    median SM clock, the maximum clock, and every throttle reason seen active.  With a
    window (start, end) of local times, only the samples taken inside it count; if none
    is, every sample does, and "window" says so."""
    rows = []
    for line in lines:
        parts = [x.strip() for x in line.split(",")]
        if len(parts) >= 10 and parts[2].isdigit():
            rows.append(parts)
    if not rows:
        return None
    where = "whole run"
    if window is not None:
        inside = [r for r in rows
                  if (t := _sample_time(r[0])) is not None and window[0] <= t <= window[1]]
        if inside:
            rows, where = inside, "timed region"
        else:
            where = "whole run (no sample fell inside the timed region)"
    sm = [int(r[2]) for r in rows]
    reasons = set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for r in rows:
        for n, v in zip(names, r[6:10]):
            if v.lower() == "active":
                reasons.add(n)
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": int(rows[0][3]),
            "samples": len(rows), "window": where, "reasons": sorted(reasons)}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def _reduce_over_ranks(x: float, world: int, op: str, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def _max_over_ranks(x: float, world: int, device=None) -> float:
    return _reduce_over_ranks(x, world, "max", device)


def job_throughput(ms_local: float, units_local: float, world: int, device=None):
    """(step ms, units/s) of the whole job: every rank runs its own replica, the step
    time is the slowest rank's and the throughput counts the units of all ranks."""
    ms_max = _reduce_over_ranks(ms_local, world, "max", device)
    units = _reduce_over_ranks(units_local, world, "sum", device)
    return ms_max, units / (ms_max / 1e3)


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ CPU oracle
def oracle_pass(wl, hd, bt, blocks):
    """One propose + verify of the oracle on the first ``blocks`` blocks."""
    from oracle import propose, verify
    from workloads import make_target
    sub = {k: v[:blocks] for k, v in bt.items()}
    o = propose(sub["hidden"], sub["anchors"], hd["lm_head"], hd["markov_w1"],
                hd["markov_w2"], L_in=wl.L_in, sample_from_anchor=wl.sample_from_anchor,
                top_k=wl.top_k, conf_min=wl.conf_min, lm_bias=hd.get("lm_bias"),
                w_conf=hd.get("w_conf"), b_conf=hd.get("b_conf", 0.0),
                topk_markov=wl.topk_markov)
    target = make_target(wl, o["draft"])
    verify(o["draft"], o["n_draft"], target)
    return o


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(wl, hd, bt, budget_s=20.0, blocks=4, min_work_s=10.0, min_passes=3):
    """Time the oracle as it stands on a bounded sample; returns the JSON object.

    Passes repeat until at least ``min_work_s`` of oracle work (and ``min_passes``
    passes) is timed, and stop before a further pass would run past ``budget_s``."""
    blocks = min(blocks, wl.B)
    times = []
    t_end = time.time() + budget_s
    while True:
        t0 = time.perf_counter()
        oracle_pass(wl, hd, bt, blocks)
        times.append(time.perf_counter() - t0)
        if time.time() + times[-1] > t_end:
            break
        if len(times) >= min_passes and sum(times) >= min_work_s:
            break
    t = statistics.median(times)
    return {"value": blocks * wl.N / t, "unit": UNIT, "cores": _cores(), "kind": "oracle",
            "sample": f"{blocks} of {wl.B} blocks x {wl.N} slots, full vocabulary "
                      f"(V={wl.V}), propose + verify, float64 NumPy; median of "
                      f"{len(times)} passes ({t:.2f} s each, {sum(times):.1f} s in all)"}


def run_reference(args):
    rank, world, local = _dist()
    if rank != 0:
        return 0
    from workloads import WORKLOADS, make_batch, make_head
    wl = WORKLOADS[args.workload]
    hd, bt = make_head(wl), make_batch(wl)
    blocks = 1
    for _ in range(args.warmup):
        oracle_pass(wl, hd, bt, blocks)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_pass(wl, hd, bt, blocks)
        times.append(time.perf_counter() - t0)
    t = sum(times) / len(times)
    v = blocks * wl.N / t
    line = {"impl": "reference", "metric": metric_of(wl), "value": v, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": _config(wl, "host cores, no L2 flush (CPU)"),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": _cores(), "kind": "oracle",
                             "sample": f"{blocks} of {wl.B} blocks per step, all {wl.N} "
                                       f"slots, full vocabulary, propose + verify"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def _config(wl, l2):
    return {"workload": wl.name, "B": wl.B, "L": wl.L_in, "N": wl.N, "H": wl.H, "V": wl.V,
            "r": wl.r, "top_k": wl.top_k, "conf_min": wl.conf_min,
            "layout": "anchor-first" if wl.sample_from_anchor else "1+N bonus anchor",
            "n_emit": wl.n_emit, "l2": l2, "parallelism": "replicas (blocks per GPU)"}


# ------------------------------------------------------------------ GPU arm
def _time_steps(tio, _abi, cfg, head, ws, hidden, anchors, out, target, acc, bonus,
                emitted, stream, flush, K, W, world, graph=False):
    """W warm-up steps, then K timed steps (L2 flushed before each, untimed): device time
    per step from CUDA events on the launching stream around dspark_propose +
    dspark_verify, called directly or (graph=True) replayed from a CUDA graph of one
    pass captured after the warm-up.  Then K more direct steps through
    dspark_propose_timed for the per-stage breakdown (its stage events add a little time
    of their own, so the step time comes from the first set)."""
    import torch
    ns = _abi.DSPARK_NUM_STAGES

    def step(events=None, s=None):
        s = stream if s is None else s
        if events is None:
            tio.propose(cfg, head, hidden, anchors, out, ws, s)
        else:
            _abi.check(_abi.dspark_propose_timed(
                cfg, head.struct(), hidden.data_ptr(), anchors.data_ptr(), out.struct(),
                ws.data_ptr(), ws.numel(), s.cuda_stream, [e.cuda_event for e in events]))
        tio.verify(out.draft, out.n_draft, target, acc, bonus, emitted, s)

    for _ in range(W):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert tio.device_status(ws, stream) == 0
    g = None
    if graph:
        # one pass captured as it is replayed by a decoding loop (same buffers)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(s=torch.cuda.current_stream())
        torch.cuda.synchronize()
    ev_step = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
    torch.cuda.synchronize()
    _barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    t_begin = datetime.datetime.now()
    for s_ in range(K):
        flush.zero_()                                   # untimed L2 flush
        ev_step[s_][0].record(stream)
        if g is not None:
            g.replay()
        else:
            step()
        ev_step[s_][1].record(stream)
    torch.cuda.synchronize()
    _barrier(world)
    t_wall = time.perf_counter() - t_wall
    window = (t_begin, datetime.datetime.now())
    assert tio.device_status(ws, stream) == 0
    step_ms = [a.elapsed_time(b) for a, b in ev_step]
    del g

    # per-stage breakdown
    ev_stage = [[torch.cuda.Event(enable_timing=True) for _ in range(ns + 1)] for _ in range(K)]
    for evs in ev_stage:          # materialise the handles the library records into
        for e in evs:
            e.record(stream)
    torch.cuda.synchronize()
    for s_ in range(K):
        flush.zero_()
        step(ev_stage[s_])
    torch.cuda.synchronize()
    assert tio.device_status(ws, stream) == 0
    stage_ms = {name: statistics.mean(ev_stage[s_][i].elapsed_time(ev_stage[s_][i + 1])
                                      for s_ in range(K))
                for i, name in enumerate(_abi.STAGE_NAMES)}
    return statistics.mean(step_ms), stage_ms, t_wall, window


def run_ours(args):
    import torch
    rank, world, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from dspark_block_drafter_gb300 import _abi
    from dspark_block_drafter_gb300 import torch_io as tio
    from workloads import WORKLOADS, make_batch, make_head, make_target

    wl = WORKLOADS[args.workload]
    hd = make_head(wl)
    bt = make_batch(wl, batch_index=rank)           # each replica drafts its own batch
    # a reduced draft vocabulary is given in its bias form (full-V head + lm_bias); the
    # prepared head holds its compact form.  The d2t form (caller-side compact head) is
    # timed beside it as an extra.
    form = "full"
    dense_head = tio.head_to_device(hd, form, dev)
    cfg = tio.make_config(wl.B, wl.L_in, wl.H, wl.V, wl.r, wl.top_k, wl.sample_from_anchor,
                          wl.conf_min, wl.dtype, wl.topk_markov)
    hidden = tio.to_device(bt["hidden"], dev)
    anchors = tio.to_device(bt["anchors"], dev)
    out = tio.Outputs.allocate(wl.B, wl.N, wl.top_k, dense_head.V_head, dev, topk=True,
                               conf=True)
    stream = torch.cuda.current_stream(dev)
    acc = torch.empty(wl.B, dtype=torch.int32, device=dev)
    bonus = torch.empty(wl.B, dtype=torch.int32, device=dev)
    emitted = torch.empty(wl.B, wl.N + 1, dtype=torch.int32, device=dev)

    # target tokens: agree with this replica's draft for a seeded geometric prefix
    ws_d = tio.workspace_for(cfg, dense_head, dev)
    tio.propose(cfg, dense_head, hidden, anchors, out, ws_d, stream)
    torch.cuda.synchronize()
    target = tio.to_device(make_target(wl, out.draft.cpu().numpy(), rank), dev)

    # the pruned chain needs the head prepared once (markov_w2 transposed + column norms),
    # like converting a checkpoint: done before timing
    head, ws, t_prep = dense_head, ws_d, None
    if args.chain == "pruned" and wl.dtype == "bf16":
        head = dataclasses.replace(dense_head)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        head.prepare(cfg, stream)
        torch.cuda.synchronize()
        t_prep = time.perf_counter() - t0
        ws = tio.workspace_for(cfg, head, dev)
    flush = L2Flush(FLUSH_BYTES, dev)
    common = (hidden, anchors, out, target, acc, bonus, emitted, stream, flush)

    K = args.steps
    clocks = ClockSampler(local if "CUDA_VISIBLE_DEVICES" not in os.environ else
                          int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local]))
    clocks.start()
    # t_pass: the pass replayed from a CUDA graph, as a decoding loop runs it
    ms, stage_ms, t_wall, window = _time_steps(tio, _abi, cfg, head, ws, *common, K,
                                               args.warmup, world, graph=True)
    clk = clocks.stop(window)
    if clk and set(clk["reasons"]) & set(BAD_CLOCK_REASONS):
        # a run the GPU throttled for heat or a hardware slowdown is no measurement:
        # take it once more and report that one
        first = clk["reasons"]
        clocks.start()
        ms, stage_ms, t_wall, window = _time_steps(tio, _abi, cfg, head, ws, *common, K,
                                                   args.warmup, world, graph=True)
        clk = clocks.stop(window)
        if clk:
            clk["remeasured_after"] = first
    ms_max, value = job_throughput(ms, wl.B * wl.N, world, dev)
    # the same pass through direct calls, beside it
    ms_d, _, _, _ = _time_steps(tio, _abi, cfg, head, ws, *common, K, args.warmup, world)
    ms_direct, _ = job_throughput(ms_d, wl.B * wl.N, world, dev)
    slots = wl.B * wl.N * world
    launches = _abi.dspark_propose_kernel_count(cfg, head.struct(), out.struct()) + 1

    # the other chain form on the same inputs, for reference
    other = None
    if head is not dense_head:
        ms_o, stage_o, _, _ = _time_steps(tio, _abi, cfg, dense_head, ws_d, *common,
                                       max(3, K // 2), args.warmup, world)
        ms_o = _max_over_ranks(ms_o, world, dev)
        other = {"chain": "dense", "value": slots / (ms_o / 1e3), "ms_per_step": ms_o,
                 "stage_us": {k: v * 1e3 for k, v in stage_o.items()}}

    # the adaptive block length (skip_truncated) on the same inputs, for reference: work
    # stops at each block's confidence cut, so it is counted in blocks and in the slots
    # actually drafted (sum of n_draft), never as B x N drafted slots
    adaptive = None
    if head is not dense_head:
        cfg_a = _abi.dspark_config.from_buffer_copy(cfg)
        cfg_a.skip_truncated = 1
        ms_a, stage_a, _, _ = _time_steps(tio, _abi, cfg_a, head, ws, *common, max(3, K // 2),
                                       args.warmup, world)
        ms_a = _max_over_ranks(ms_a, world, dev)
        drafted = int(out.n_draft.sum().item())
        adaptive = {"skip_truncated": 1, "ms_per_step": ms_a,
                    "verified_blocks_per_s": wl.B * world / (ms_a / 1e3),
                    "drafted_slots_per_s": drafted * world / (ms_a / 1e3),
                    "mean_n_draft": drafted / wl.B,
                    "stage_us": {k: v * 1e3 for k, v in stage_a.items()}}

    # end to end through the host-buffer entry point (copies inside the timed region)
    e2e = e2e_host(cfg, head, wl, bt, target, dev, stream, flush, K, args.warmup, world)

    # dspark_verify alone, back to back on this GPU (an extra; never the headline)
    verify_only = _verify_only(tio, out, target, acc, bonus, emitted, stream, K,
                               args.warmup, wl.B)

    # the pruned chain where its bounds are loose (an extra; never the headline)
    loose = None
    if head is not dense_head and wl.name == "qwen3_8b_b32":
        loose = _loose_markov(tio, wl, hd, form, cfg, dev, common, max(3, K // 4),
                              args.warmup, world)

    # the d2t form of a reduced vocabulary, for comparison (an extra)
    d2t_form = None
    if wl.n_emit and head is not dense_head:
        d2t_form = _d2t_form(tio, _abi, wl, hd, cfg, dev, common, max(3, K // 2), args.warmup,
                             world)

    peaks = _peaks()
    # (the algorithmic work of a reduced vocabulary is over its emittable rows)
    alg = _algorithmic(wl, wl.n_emit or head.V_head)
    gemm_ms = stage_ms["logits"]
    compute_tf = peaks["bf16_tflops"] if wl.dtype == "bf16" else FP32_ALU_TFLOPS
    t_roof = max(alg["bytes"] / (peaks["hbm_gbs"] * 1e9),
                 alg["flops"] / (compute_tf * 1e12))
    # the GEMM's own bound: whichever of its bytes and flops takes longer at peak
    if alg["gemm_bytes"] / (peaks["hbm_gbs"] * 1e9) > alg["gemm_flops"] / (compute_tf * 1e12):
        bound, unit, peak = "hbm", "GB/s", peaks["hbm_gbs"]
        achieved = alg["gemm_bytes"] / (gemm_ms / 1e3) / 1e9
        peak_source = f"{peaks['_source']} HBM copy"
    else:
        bound = "tensor" if wl.dtype == "bf16" else "alu"
        unit, peak = "TFLOP/s", compute_tf
        achieved = alg["gemm_flops"] / (gemm_ms / 1e3) / 1e12
        peak_source = (f"{peaks['_source']} bf16 burst" if wl.dtype == "bf16" else
                       "fp32 lanes x clock (derived)")
    line = {
        "metric": metric_of(wl), "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
        "config": _config(wl, f"flushed: {FLUSH_BYTES >> 20} MB written, then another "
                              f"{FLUSH_BYTES >> 20} MB read, before each timed "
                              "step (untimed)"),
        "verified_blocks_per_s": wl.B * world / (ms_max / 1e3),
        "t_pass_us": ms_max * 1e3,
        "timing": "CUDA-graph replay of one pass (dspark_propose + dspark_verify)",
        "t_pass_direct_us": ms_direct * 1e3,
        "stage_us": {k: v * 1e3 for k, v in stage_ms.items()},
        "chain": "pruned" if head is not dense_head else "dense",
        "head_prepare_ms": None if t_prep is None else t_prep * 1e3,
        "pass_roofline": {"t_roof_us": t_roof * 1e6, "frac": t_roof / (ms_max / 1e3),
                          "bytes": alg["bytes"], "flops": alg["flops"],
                          "peaks": peaks["_source"]},
        "roofline": {"kernel": "base logits (lm_head GEMM)", "bound": bound,
                     "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak,
                     "traffic": GEMM_TRAFFIC.get(wl.name, (None, None))[0],
                     "traffic_source": GEMM_TRAFFIC.get(wl.name, (None, None))[1],
                     "algorithmic_bytes": alg["gemm_bytes"],
                     "peak_source": peak_source},
        "e2e": e2e,
        "gpu_launches": K * launches,
        "other_chain": other,
        "adaptive": adaptive,
        "loose_markov": loose,
        "d2t_form": d2t_form,
        "verify_only": verify_only,
        "clocks": clk,
        "wall_s_timed_region": t_wall,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, hd, bt)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def _d2t_form(tio, _abi, wl, hd, cfg, dev, common, K, W, world):
    """The same batch with the reduced vocabulary as a compact head + d2t table built by
    the caller (the form the bias form is compacted into by dspark_prepare_head)."""
    import torch
    head = tio.head_to_device(hd, "d2t", dev)
    head.prepare(cfg, common[7])
    ws = tio.workspace_for(cfg, head, dev)
    ms, stage, _, _ = _time_steps(tio, _abi, cfg, head, ws, *common, K, W, world)
    res = {"ms_per_step": _max_over_ranks(ms, world, dev),
           "stage_us": {k: v * 1e3 for k, v in stage.items()}}
    del ws, head
    torch.cuda.empty_cache()
    return res


def _loose_markov(tio, wl, hd, form, cfg, dev, common, K, W, world, std=0.3):
    """The same head and batch with markov_w1, markov_w2 ~ N(0, std): at 0.3 the Markov
    term spreads about as widely as the logits (std 16 x 0.3^2 = 1.44 against 1.28), so
    the pruned chain's Cauchy-Schwarz bounds admit many rows.  Pass time of both chain
    forms, and how many (slot, block) pairs the pruned walk evaluated on the fly."""
    import torch
    from workloads import make_markov
    from dspark_block_drafter_gb300 import _abi
    w1, w2 = make_markov(dataclasses.replace(wl, markov_std=std))
    hd_l = dict(hd, markov_w1=w1, markov_w2=w2)
    dense = tio.head_to_device(hd_l, form, dev)
    pruned = dataclasses.replace(dense)
    stream = common[7]
    pruned.prepare(cfg, stream)
    res = {"markov_std": std, "slots": wl.B * wl.N}
    for name, head in (("pruned", pruned), ("dense", dense)):
        ws = tio.workspace_for(cfg, head, dev)
        ms, stage, _, _ = _time_steps(tio, _abi, cfg, head, ws, *common, K, W, world)
        st = tio.pass_stats(ws, stream)
        res[name] = {"ms_per_step": _max_over_ranks(ms, world, dev),
                     "stage_us": {k: v * 1e3 for k, v in stage.items()}, **st}
        del ws
    res["pruned"]["share_on_the_fly"] = res["pruned"]["on_the_fly"] / (wl.B * wl.N)
    del dense, pruned
    torch.cuda.empty_cache()
    return res


def _verify_only(tio, out, target, acc, bonus, emitted, stream, K, W, B):
    """Device time of dspark_verify alone (K calls back to back after W warm-up calls, on
    the proposal's draft): per call and as verified blocks/s of this GPU.  Any failure
    leaves the extra out (None) instead of ending the benchmark."""
    import torch
    try:
        for _ in range(W):
            tio.verify(out.draft, out.n_draft, target, acc, bonus, emitted, stream)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            tio.verify(out.draft, out.n_draft, target, acc, bonus, emitted, stream)
        e1.record(stream)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / K
        return {"us_per_call": us, "blocks_per_s": B / (us * 1e-6), "calls": K}
    except Exception as exc:  # an extra: report why it is missing, keep the line
        return {"unavailable": f"{type(exc).__name__}: {exc}"}


def e2e_host(cfg, head, wl, bt, target_dev, dev, stream, flush, K, W, world):
    """Same metric through dspark_step_host with page-locked host buffers."""
    import torch
    from dspark_block_drafter_gb300 import _abi
    from dspark_block_drafter_gb300 import torch_io as tio
    hidden_h = tio.to_device(bt["hidden"], "cpu").pin_memory()
    anchors_h = torch.from_numpy(bt["anchors"]).pin_memory()
    target_h = target_dev.cpu().pin_memory()
    B, N, k = wl.B, wl.N, wl.top_k
    i32 = dict(dtype=torch.int32, pin_memory=True)
    draft_h, nd_h = torch.empty(B, N, **i32), torch.empty(B, **i32)
    acc_h, bon_h = torch.empty(B, **i32), torch.empty(B, **i32)
    tki_h = torch.empty(B, N, k, **i32)
    tkv_h = torch.empty(B, N, k, dtype=torch.float32, pin_memory=True)
    n = _abi.dspark_step_host_workspace_size(cfg, head.struct())
    ws = torch.empty(n, dtype=torch.uint8, device=dev)

    def go():
        _abi.check(_abi.dspark_step_host(cfg, head.struct(), hidden_h.data_ptr(),
                                         anchors_h.data_ptr(), target_h.data_ptr(),
                                         draft_h.data_ptr(), nd_h.data_ptr(), acc_h.data_ptr(),
                                         bon_h.data_ptr(), tki_h.data_ptr(), tkv_h.data_ptr(),
                                         ws.data_ptr(), n, stream.cuda_stream))
    for _ in range(W):
        flush.zero_()
        go()
    torch.cuda.synchronize()
    times = []
    for _ in range(K):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        go()
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b))
    ms = _max_over_ranks(statistics.mean(times), world, dev)
    h2d = hidden_h.numel() * hidden_h.element_size() + 4 * B + 4 * B * (N + 1)
    d2h = 4 * (B * N + 3 * B) + 8 * B * N * k
    return {"value": B * N * world / (ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "api": "dspark_step_host (page-locked host buffers)"}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen3_8b_b32")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--chain", choices=["pruned", "dense"], default="pruned",
                    help="pruned: exact-bound pruned chain (prepared head); dense: every row")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
