"""Shared driver of the GPU parity tests: run a workload through the C ABI and through
the oracle on the same seeded inputs, then apply the tolerance checker."""
from __future__ import annotations

import numpy as np

from oracle import check, propose as oracle_propose
from workloads import make_batch, make_head

TOL = {"f32": 1e-5, "bf16": 2e-2}


def gpu_propose(wl, hd, bt, form="full", want_logits=False, want_topk=True, stream=None,
                chain="dense", skip_truncated=False, conf_hidden=None):
    """Run dspark_propose on the GPU; returns (numpy outputs, workspace tensor).

    chain "dense" evaluates every head row; "pruned" prepares the head first so that the
    exact-bound pruned chain runs (it needs the logits output off).
    """
    import torch
    from dspark_block_drafter_gb300 import torch_io as tio
    cfg = tio.make_config(wl.B, wl.L_in, wl.H, wl.V, wl.r, wl.top_k, wl.sample_from_anchor,
                          wl.conf_min, wl.dtype, wl.topk_markov, skip_truncated)
    head = tio.head_to_device(hd, form)
    if chain == "pruned":
        assert not want_logits
        head.prepare(cfg)
    hidden = tio.to_device(bt["hidden"])
    anchors = tio.to_device(bt["anchors"])
    out = tio.Outputs.allocate(wl.B, wl.N, wl.top_k, head.V_head, topk=want_topk,
                               conf=hd.get("w_conf") is not None, logits=want_logits)
    ws = tio.workspace_for(cfg, head)
    ch = None if conf_hidden is None else tio.to_device(conf_hidden)
    tio.propose(cfg, head, hidden, anchors, out, ws, stream, conf_hidden=ch)
    torch.cuda.synchronize()
    st = tio.device_status(ws)
    assert st == 0, f"device status {st}"
    return out.numpy(), ws


def oracle_run(wl, hd, bt, want_logits=False, skip_truncated=False, conf_hidden=None):
    return oracle_propose(bt["hidden"], bt["anchors"], hd["lm_head"], hd["markov_w1"],
                          hd["markov_w2"], L_in=wl.L_in,
                          sample_from_anchor=wl.sample_from_anchor, top_k=wl.top_k,
                          conf_min=wl.conf_min, lm_bias=hd.get("lm_bias"),
                          w_conf=hd.get("w_conf"), b_conf=hd.get("b_conf", 0.0),
                          topk_markov=wl.topk_markov, return_logits=want_logits,
                          skip_truncated=skip_truncated, conf_hidden=conf_hidden)


def compare(wl, hd, bt, o, g, form="full", skip_truncated=False):
    head_rows = hd["emit_rows"] if form == "d2t" else None
    rep = check.check_propose(o, anchors=bt["anchors"], markov_w1=hd["markov_w1"],
                              markov_w2=hd["markov_w2"], top_k=wl.top_k,
                              topk_markov=wl.topk_markov, conf_min=wl.conf_min,
                              gpu=g, tol=TOL[wl.dtype], head_rows=head_rows,
                              lm_bias=hd.get("lm_bias"), skip_truncated=skip_truncated)
    return rep


def run_case(wl, form="full", want_logits=True, hd=None, bt=None, chain="dense",
             skip_truncated=False, conf_hidden=None):
    hd = make_head(wl) if hd is None else hd
    bt = make_batch(wl) if bt is None else bt
    g, _ = gpu_propose(wl, hd, bt, form, want_logits and chain == "dense", chain=chain,
                       skip_truncated=skip_truncated, conf_hidden=conf_hidden)
    o = oracle_run(wl, hd, bt, skip_truncated=skip_truncated, conf_hidden=conf_hidden)
    rep = compare(wl, hd, bt, o, g, form, skip_truncated=skip_truncated)
    assert rep["failures"] == [], rep
    return g, o, rep
