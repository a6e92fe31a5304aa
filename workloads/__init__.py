"""Seeded synthetic inputs for the DSpark proposal head and the greedy verify step.

This module holds shapes and random draws only; none of the method's arithmetic lives
here.  Both the CPU oracle and the CUDA path read the arrays it returns, and neither
of them is imported from here.

Every array is drawn from NumPy's PCG64 with one sub-stream per tensor (and per row
chunk for the large ones), so a workload is reproducible bit for bit on any host.
Floating-point values are drawn in fp32; for the bf16 workloads they are rounded to
bf16 with round-to-nearest-even and handed out as raw ``uint16`` bit patterns, so the
two sides upcast the very same bits.

Workload shapes follow the heads the DSpark pages talk about: a Qwen3-8B-shaped
head (H=4096, V=151936), a Qwen3.8-27B-shaped head (H=5120, V=248320, mask token
248077 from lucebox PR #626's loader notes) and a Gemma-4-shaped reduced-vocabulary
head in the 1+N bonus-anchor layout (llama.cpp PR #26275, the speculators-format
description).  No checkpoint, prompt or dataset is involved.
"""
from __future__ import annotations

import dataclasses
from concurrent.futures import ThreadPoolExecutor
from typing import Optional

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "make_head", "make_batch", "make_target",
    "make_conf_hidden", "make_lattice_target", "to_bf16_bits", "slots_of",
]

# sub-stream ids, one per tensor
(_S_LM_HEAD, _S_W1, _S_W2, _S_WCONF, _S_HIDDEN, _S_ANCHORS, _S_EMIT, _S_TARGET,
 _S_CONF_HIDDEN, _S_LATTICE) = range(1, 11)
_ROW_CHUNK = 4096


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape and value recipe of one synthetic DSpark head + batch."""
    name: str
    B: int                      # blocks in the batch
    L_in: int                   # slots per block in the hidden-state tensor
    H: int                      # hidden size
    V: int                      # vocabulary size
    r: int                      # Markov rank
    top_k: int                  # candidates kept per prediction slot
    sample_from_anchor: bool    # True: anchor-first; False: 1+N bonus anchor
    conf_min: float             # truncation threshold (<= 0 disables)
    dtype: str                  # "f32" or "bf16"
    weight_std: float           # std of lm_head, markov_w1, markov_w2
    conf_std: float             # std of w_conf
    b_conf: float = 0.0
    n_emit: Optional[int] = None      # emittable rows (others get a -1e9 bias)
    mask_token: Optional[int] = None  # never drawn as an anchor
    topk_markov: bool = True          # top-k over corrected (True) or base logits
    accept_p: Optional[float] = None  # per-slot mismatch probability of the target;
                                      # None: exactly one mismatch per block
    seed: int = 20260
    markov_std: Optional[float] = None  # std of markov_w1 and markov_w2 (None: weight_std)

    @property
    def N(self) -> int:
        """Prediction slots per block."""
        return self.L_in if self.sample_from_anchor else self.L_in - 1

    @property
    def M(self) -> int:
        return self.B * self.N

    def scaled(self, **kw) -> "Workload":
        """Same recipe with some sizes replaced (used for small parity cases)."""
        name = kw.pop("name", self.name + "-scaled")
        return dataclasses.replace(self, name=name, **kw)


def slots_of(wl: Workload) -> tuple[int, int]:
    """(N, i_first_pred) of a workload's block layout."""
    return (wl.L_in, 0) if wl.sample_from_anchor else (wl.L_in - 1, 1)


WORKLOADS: dict[str, Workload] = {
    w.name: w for w in [
        Workload("tiny_fp32", B=2, L_in=4, H=256, V=4096, r=16, top_k=4,
                 sample_from_anchor=True, conf_min=0.0, dtype="f32",
                 weight_std=0.05, conf_std=0.05, accept_p=None, seed=20260),
        Workload("qwen3_8b_b1", B=1, L_in=16, H=4096, V=151936, r=256, top_k=1,
                 sample_from_anchor=True, conf_min=0.0, dtype="bf16",
                 weight_std=0.02, conf_std=0.02, accept_p=0.5, seed=20261),
        Workload("qwen3_8b_b32", B=32, L_in=16, H=4096, V=151936, r=256, top_k=8,
                 sample_from_anchor=True, conf_min=0.5, dtype="bf16",
                 weight_std=0.02, conf_std=0.02, accept_p=0.4, seed=20262),
        Workload("qwen38_27b_b8", B=8, L_in=16, H=5120, V=248320, r=256, top_k=8,
                 sample_from_anchor=True, conf_min=0.3, dtype="bf16",
                 weight_std=0.02, conf_std=0.02, mask_token=248077,
                 accept_p=0.5, seed=20263),
        Workload("gemma4_bonus_b64", B=64, L_in=7, H=2816, V=262144, r=128, top_k=1,
                 sample_from_anchor=False, conf_min=0.5, dtype="bf16",
                 weight_std=0.02, conf_std=0.02, n_emit=32768,
                 accept_p=0.46, seed=20264),
    ]
}


def _rng(seed: int, *stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *stream])))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even); returns uint16 bit patterns.

    Input quantisation of the synthetic draws, identical to torch's fp32 -> bf16
    conversion for finite values.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def _normal_rows(seed: int, stream: int, rows: int, cols: int, std: float,
                 dtype: str, threads: int = 8) -> np.ndarray:
    """rows x cols N(0, std^2) draws, one sub-stream per chunk of rows."""
    out = np.empty((rows, cols), np.uint16 if dtype == "bf16" else np.float32)

    def fill(c0: int) -> None:
        c1 = min(rows, c0 + _ROW_CHUNK)
        g = _rng(seed, stream, c0 // _ROW_CHUNK)
        tmp = g.standard_normal((c1 - c0, cols), dtype=np.float32)
        tmp *= np.float32(std)
        out[c0:c1] = to_bf16_bits(tmp) if dtype == "bf16" else tmp

    starts = list(range(0, rows, _ROW_CHUNK))
    if len(starts) == 1 or threads <= 1:
        for s in starts:
            fill(s)
    else:
        with ThreadPoolExecutor(threads) as ex:
            list(ex.map(fill, starts))
    return out


def make_head(wl: Workload, threads: int = 8) -> dict:
    """The drafter head's weights.

    Returns a dict with
      lm_head   [V, H]   (uint16 bf16 bits or float32)
      markov_w1 [V, r]
      markov_w2 [r, V]
      w_conf    [H]
      b_conf    float
      lm_bias   [V] float32 or None   (0 on emittable rows, -1e9 elsewhere)
      emit_rows [n_emit] int32 sorted, or None
    """
    lm_head = _normal_rows(wl.seed, _S_LM_HEAD, wl.V, wl.H, wl.weight_std, wl.dtype, threads)
    w1, w2 = make_markov(wl, threads)
    w_conf = _normal_rows(wl.seed, _S_WCONF, 1, wl.H, wl.conf_std, wl.dtype, 1)[0]
    lm_bias = emit = None
    if wl.n_emit is not None:
        g = _rng(wl.seed, _S_EMIT)
        emit = np.sort(g.choice(wl.V, size=wl.n_emit, replace=False)).astype(np.int32)
        lm_bias = np.full(wl.V, -1e9, np.float32)
        lm_bias[emit] = 0.0
    return dict(lm_head=lm_head, markov_w1=w1, markov_w2=w2, w_conf=w_conf,
                b_conf=float(wl.b_conf), lm_bias=lm_bias, emit_rows=emit)


def make_markov(wl: Workload, threads: int = 8):
    """markov_w1 [V, r] and markov_w2 [r, V] of the head (std markov_std, else weight_std)."""
    std = wl.weight_std if wl.markov_std is None else wl.markov_std
    w1 = _normal_rows(wl.seed, _S_W1, wl.V, wl.r, std, wl.dtype, threads)
    w2 = _normal_rows(wl.seed, _S_W2, wl.r, wl.V, std, wl.dtype, threads)
    return w1, w2


def make_batch(wl: Workload, batch_index: int = 0) -> dict:
    """One batch of drafter outputs: hidden [B, L_in, H] (N(0,1)) and anchors [B].

    Anchors are uniform over [0, V) minus the mask token when the workload names one.
    """
    hidden = _normal_rows(wl.seed + 1000 * batch_index, _S_HIDDEN, wl.B * wl.L_in, wl.H,
                          1.0, wl.dtype, 8).reshape(wl.B, wl.L_in, wl.H)
    g = _rng(wl.seed + 1000 * batch_index, _S_ANCHORS)
    if wl.mask_token is None:
        anchors = g.integers(0, wl.V, size=wl.B)
    else:
        anchors = g.integers(0, wl.V - 1, size=wl.B)
        anchors = anchors + (anchors >= wl.mask_token)   # skip the mask token
    return dict(hidden=hidden, anchors=anchors.astype(np.int32))


def make_target(wl: Workload, draft: np.ndarray, batch_index: int = 0) -> np.ndarray:
    """Target-model argmax tokens [B, N+1] for the verify step.

    The target agrees with ``draft`` on a seeded prefix: with ``accept_p`` set, the
    prefix length is geometric (NumPy's ``geometric(p) - 1``: the count of agreeing
    slots before the first disagreement); without it, exactly one slot per block
    (uniform over [0, N)) disagrees.  The disagreeing slot gets a token that differs
    from the draft's; every slot after it, and the bonus slot N, is uniform.
    """
    draft = np.asarray(draft, dtype=np.int64)
    B, N = draft.shape
    g = _rng(wl.seed + 1000 * batch_index, _S_TARGET)
    target = g.integers(0, wl.V, size=(B, N + 1))
    if wl.accept_p is None:
        agree = g.integers(0, N, size=B)
    else:
        agree = g.geometric(wl.accept_p, size=B) - 1
    shift = g.integers(1, wl.V, size=B)
    for b in range(B):
        a = int(min(agree[b], N))
        target[b, :a] = draft[b, :a]
        if a < N:
            target[b, a] = (draft[b, a] + shift[b]) % wl.V
    return target.astype(np.int32)


def make_conf_hidden(wl: Workload, batch_index: int = 0) -> np.ndarray:
    """A separate input of the confidence head, [B, L_in, H], N(0, 1) like the hidden
    states but drawn from a sub-stream of its own."""
    return _normal_rows(wl.seed + 1000 * batch_index, _S_CONF_HIDDEN, wl.B * wl.L_in, wl.H,
                        1.0, wl.dtype, 8).reshape(wl.B, wl.L_in, wl.H)


def make_lattice_target(wl: Workload, topk_ids: np.ndarray, batch_index: int = 0,
                        p: Optional[float] = None) -> np.ndarray:
    """Target argmax tokens [B, N+1] for verifying a candidate lattice topk_ids [B, N, k].

    Along a seeded prefix (geometric length with mismatch probability p, default the
    workload's accept_p or 0.5) the target's token at each slot is one of that slot's
    candidates, at a uniformly drawn rank; at the end of the prefix it is a token that is
    none of the slot's candidates; every later slot and the bonus slot are uniform.
    """
    ids = np.asarray(topk_ids, np.int64)
    B, N, k = ids.shape
    g = _rng(wl.seed + 1000 * batch_index, _S_LATTICE)
    target = g.integers(0, wl.V, size=(B, N + 1))
    p = p if p is not None else (wl.accept_p if wl.accept_p is not None else 0.5)
    agree = g.geometric(p, size=B) - 1
    ranks = g.integers(0, k, size=(B, N))
    for b in range(B):
        a = int(min(agree[b], N))
        target[b, :a] = ids[b, np.arange(a), ranks[b, :a]]
        if a < N:
            x = int(g.integers(0, wl.V))
            while x in set(ids[b, a].tolist()):
                x = (x + 1) % wl.V
            target[b, a] = x
    return target.astype(np.int32)
