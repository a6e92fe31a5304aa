"""Marshalling between torch tensors and the C ABI.

PyTorch only provides device memory and streams here; the calls go straight to
libdspark.so through :mod:`._abi`.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

from . import _abi

_DT = {"f32": _abi.DSPARK_F32, "bf16": _abi.DSPARK_BF16}


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def to_device(a, device="cuda") -> torch.Tensor:
    """numpy -> device tensor; uint16 arrays are bf16 bit patterns."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def make_config(B, L_in, H, V, r, top_k, sample_from_anchor, conf_min, dtype,
                topk_markov=True, skip_truncated=False) -> _abi.dspark_config:
    return _abi.dspark_config(B=B, L_in=L_in, H=H, V=V, r=r, top_k=top_k,
                              sample_from_anchor=int(bool(sample_from_anchor)),
                              topk_markov=int(bool(topk_markov)), conf_min=float(conf_min),
                              dtype=_DT[dtype] if isinstance(dtype, str) else int(dtype),
                              skip_truncated=int(bool(skip_truncated)))


@dataclasses.dataclass
class Head:
    """Device copies of a drafter head and the matching dspark_head struct."""
    lm_head: torch.Tensor
    markov_w1: torch.Tensor
    markov_w2: torch.Tensor
    lm_bias: Optional[torch.Tensor] = None
    d2t: Optional[torch.Tensor] = None
    w_conf: Optional[torch.Tensor] = None
    b_conf: float = 0.0
    prepared: Optional[torch.Tensor] = None

    @property
    def V_head(self) -> int:
        return int(self.lm_head.shape[0])

    def struct(self) -> _abi.dspark_head:
        return _abi.dspark_head(lm_head=_ptr(self.lm_head), lm_bias=_ptr(self.lm_bias),
                                d2t=_ptr(self.d2t), V_head=self.V_head,
                                markov_w1=_ptr(self.markov_w1),
                                markov_w2=_ptr(self.markov_w2), w_conf=_ptr(self.w_conf),
                                b_conf=float(self.b_conf), prepared=_ptr(self.prepared))

    def prepare(self, cfg, stream=None) -> "Head":
        """Fill ``prepared`` with dspark_prepare_head (enables the pruned chain)."""
        bare = dataclasses.replace(self, prepared=None)
        n = _abi.dspark_prepare_head_size(cfg, bare.struct())
        if n == 0:
            _abi.check(_abi.DSPARK_ERR_UNSUPPORTED)
        buf = torch.empty(n, dtype=torch.uint8, device=self.lm_head.device)
        _abi.check(_abi.dspark_prepare_head(cfg, bare.struct(), buf.data_ptr(), n,
                                            _stream(stream)))
        self.prepared = buf
        return self


def head_to_device(h: dict, form: str = "full", device="cuda") -> Head:
    """Upload a head dict of ``workloads.make_head``.

    form "full": lm_head / markov_w2 over the whole vocabulary (+ lm_bias if any);
    form "d2t": the compact head of the emittable rows plus the d2t table (the
    reduced-vocabulary form of llama.cpp PR #26275); the gather is done here on the host.
    """
    w_conf = None if h.get("w_conf") is None else to_device(h["w_conf"], device)
    if form == "full":
        return Head(to_device(h["lm_head"], device), to_device(h["markov_w1"], device),
                    to_device(h["markov_w2"], device),
                    None if h.get("lm_bias") is None else to_device(h["lm_bias"], device),
                    None, w_conf, h.get("b_conf", 0.0))
    if form == "d2t":
        rows = h["emit_rows"]
        return Head(to_device(h["lm_head"][rows], device), to_device(h["markov_w1"], device),
                    to_device(np.ascontiguousarray(h["markov_w2"][:, rows]), device),
                    to_device(h["lm_bias"][rows], device),
                    to_device(rows.astype(np.int32), device), w_conf, h.get("b_conf", 0.0))
    raise ValueError(form)


@dataclasses.dataclass
class Outputs:
    draft: torch.Tensor
    n_draft: torch.Tensor
    topk_ids: Optional[torch.Tensor] = None
    topk_vals: Optional[torch.Tensor] = None
    conf: Optional[torch.Tensor] = None
    logits: Optional[torch.Tensor] = None

    @classmethod
    def allocate(cls, B, N, k, V_head, device="cuda", topk=True, conf=True, logits=False):
        i32 = dict(dtype=torch.int32, device=device)
        f32 = dict(dtype=torch.float32, device=device)
        return cls(torch.empty(B, N, **i32), torch.empty(B, **i32),
                   torch.empty(B, N, k, **i32) if topk else None,
                   torch.empty(B, N, k, **f32) if topk else None,
                   torch.empty(B, N, **f32) if conf else None,
                   torch.empty(B, N, V_head, **f32) if logits else None)

    def struct(self) -> _abi.dspark_outputs:
        return _abi.dspark_outputs(draft=_ptr(self.draft), n_draft=_ptr(self.n_draft),
                                   topk_ids=_ptr(self.topk_ids), topk_vals=_ptr(self.topk_vals),
                                   conf=_ptr(self.conf), logits=_ptr(self.logits))

    def numpy(self) -> dict:
        return {k: (None if v is None else v.cpu().numpy())
                for k, v in dataclasses.asdict(self).items()}


def workspace_for(cfg, head: Head, device="cuda") -> torch.Tensor:
    n = _abi.dspark_propose_workspace_size(cfg, head.struct())
    if n == 0:
        _abi.check(_abi.DSPARK_ERR_INVALID_ARG)
    return torch.empty(n, dtype=torch.uint8, device=device)


def propose(cfg, head: Head, hidden: torch.Tensor, anchors: torch.Tensor, out: Outputs,
            workspace: torch.Tensor, stream=None, conf_hidden: Optional[torch.Tensor] = None
            ) -> None:
    """dspark_propose on torch tensors; raises DSparkError on a non-OK status."""
    _abi.check(_abi.dspark_propose(cfg, head.struct(), hidden.data_ptr(), anchors.data_ptr(),
                                   out.struct(), workspace.data_ptr(), workspace.numel(),
                                   _stream(stream), _ptr(conf_hidden)))


def verify(draft, n_draft, target, accepted, bonus, emitted=None, stream=None) -> None:
    """dspark_verify on torch tensors; raises DSparkError on a non-OK status."""
    B, N = draft.shape
    _abi.check(_abi.dspark_verify(B, N, draft.data_ptr(), n_draft.data_ptr(),
                                  target.data_ptr(), accepted.data_ptr(), bonus.data_ptr(),
                                  _ptr(emitted), _stream(stream)))


def tree_verify(topk_ids, n_draft, target, accepted, bonus, emitted=None, path=None,
                stream=None) -> None:
    """dspark_tree_verify on torch tensors; raises DSparkError on a non-OK status."""
    B, N, k = topk_ids.shape
    _abi.check(_abi.dspark_tree_verify(B, N, k, topk_ids.data_ptr(), n_draft.data_ptr(),
                                       target.data_ptr(), accepted.data_ptr(),
                                       bonus.data_ptr(), _ptr(emitted), _ptr(path),
                                       _stream(stream)))


def device_status(workspace: torch.Tensor, stream=None) -> int:
    return _abi.dspark_device_status(workspace.data_ptr(), _stream(stream))


def pass_stats(workspace: torch.Tensor, stream=None) -> dict:
    return _abi.dspark_pass_stats(workspace.data_ptr(), _stream(stream))
