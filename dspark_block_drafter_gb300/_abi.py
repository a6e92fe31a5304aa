"""ctypes binding of libdspark.so: the C ABI of include/dspark.h, one Python function
per C entry point, with the same names.  Argument marshalling only; every step of the
proposal and of verify runs in the library's CUDA kernels.

Pointers are passed as Python ints (device addresses, e.g. ``tensor.data_ptr()``);
``stream`` is a cudaStream_t as an int (0 = legacy default stream).
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdspark.so")

DSPARK_OK = 0
DSPARK_ERR_INVALID_ARG = 1
DSPARK_ERR_UNSUPPORTED = 2
DSPARK_ERR_WORKSPACE = 3
DSPARK_ERR_CUDA = 4
DSPARK_ERR_DEVICE = 5
DSPARK_ERR_TIMEOUT = 6
DSPARK_F32 = 0
DSPARK_BF16 = 1

c_i32 = ctypes.c_int32
c_ptr = ctypes.c_void_p


class dspark_config(ctypes.Structure):
    _fields_ = [("B", c_i32), ("L_in", c_i32), ("H", c_i32), ("V", c_i32), ("r", c_i32),
                ("top_k", c_i32), ("sample_from_anchor", c_i32), ("topk_markov", c_i32),
                ("conf_min", ctypes.c_float), ("dtype", c_i32), ("skip_truncated", c_i32)]


class dspark_head(ctypes.Structure):
    _fields_ = [("lm_head", c_ptr), ("lm_bias", c_ptr), ("d2t", c_ptr), ("V_head", c_i32),
                ("markov_w1", c_ptr), ("markov_w2", c_ptr), ("w_conf", c_ptr),
                ("b_conf", ctypes.c_float), ("prepared", c_ptr)]


class dspark_outputs(ctypes.Structure):
    _fields_ = [("draft", c_ptr), ("n_draft", c_ptr), ("topk_ids", c_ptr),
                ("topk_vals", c_ptr), ("conf", c_ptr), ("logits", c_ptr)]


class DSparkError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"dspark status {status}: {message}")
        self.status = status


_lib = None

# name -> (restype, argtypes) for every symbol include/dspark.h declares
SIGNATURES = {
    "dspark_num_slots": (c_i32, [ctypes.POINTER(dspark_config)]),
    "dspark_propose_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(dspark_config),
                                                        ctypes.POINTER(dspark_head)]),
    "dspark_propose": (c_i32, [ctypes.POINTER(dspark_config), ctypes.POINTER(dspark_head),
                               c_ptr, c_ptr, c_ptr, ctypes.POINTER(dspark_outputs), c_ptr,
                               ctypes.c_size_t, c_ptr]),
    "dspark_propose_timed": (c_i32, [ctypes.POINTER(dspark_config),
                                     ctypes.POINTER(dspark_head), c_ptr, c_ptr, c_ptr,
                                     ctypes.POINTER(dspark_outputs), c_ptr, ctypes.c_size_t,
                                     c_ptr, ctypes.POINTER(c_ptr)]),
    "dspark_propose_kernel_count": (c_i32, [ctypes.POINTER(dspark_config),
                                            ctypes.POINTER(dspark_head),
                                            ctypes.POINTER(dspark_outputs)]),
    "dspark_step_host_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(dspark_config),
                                                          ctypes.POINTER(dspark_head)]),
    "dspark_step_host": (c_i32, [ctypes.POINTER(dspark_config), ctypes.POINTER(dspark_head),
                                 c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr,
                                 c_ptr, c_ptr, c_ptr, ctypes.c_size_t, c_ptr]),
    "dspark_prepare_head_size": (ctypes.c_size_t, [ctypes.POINTER(dspark_config),
                                                   ctypes.POINTER(dspark_head)]),
    "dspark_prepare_head": (c_i32, [ctypes.POINTER(dspark_config), ctypes.POINTER(dspark_head),
                                    c_ptr, ctypes.c_size_t, c_ptr]),
    "dspark_propose_noalloc": (c_i32, [ctypes.POINTER(dspark_config),
                                       ctypes.POINTER(dspark_head), c_ptr, c_ptr, c_ptr,
                                       ctypes.POINTER(dspark_outputs), c_ptr]),
    "dspark_verify": (c_i32, [c_i32, c_i32, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr]),
    "dspark_tree_verify": (c_i32, [c_i32, c_i32, c_i32, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr,
                                   c_ptr, c_ptr, c_ptr]),
    "dspark_device_status": (c_i32, [c_ptr, c_ptr]),
    "dspark_noalloc_device_status": (c_i32, [c_ptr]),
    "dspark_pass_stats": (c_i32, [c_ptr, c_ptr, ctypes.POINTER(c_i32), ctypes.POINTER(c_i32),
                                  ctypes.POINTER(c_i32)]),
    "dspark_wait_selftest": (c_i32, [c_ptr, ctypes.c_size_t, ctypes.c_int64, c_i32, c_ptr]),
    "dspark_status_string": (ctypes.c_char_p, [c_i32]),
    "dspark_last_error": (ctypes.c_char_p, []),
}


def lib() -> ctypes.CDLL:
    """The loaded library.  Raises if it has not been built: there is no other path."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing; build it with "
                "`python -m dspark_block_drafter_gb300.build`")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib = l
    return _lib


def check(status: int) -> None:
    """Raise DSparkError for a non-OK status, with the library's message."""
    if status != DSPARK_OK:
        msg = dspark_last_error() or dspark_status_string(status)
        raise DSparkError(status, msg)


def dspark_num_slots(cfg: dspark_config) -> int:
    return lib().dspark_num_slots(ctypes.byref(cfg))


def dspark_propose_workspace_size(cfg: dspark_config, head: dspark_head) -> int:
    return lib().dspark_propose_workspace_size(ctypes.byref(cfg), ctypes.byref(head))


def dspark_propose(cfg: dspark_config, head: dspark_head, hidden: int, anchors: int,
                   out: dspark_outputs, workspace: int, workspace_bytes: int,
                   stream: int = 0, conf_hidden: int | None = None) -> int:
    """``conf_hidden`` goes to the C argument of that name (after ``anchors``)."""
    return lib().dspark_propose(ctypes.byref(cfg), ctypes.byref(head), hidden, anchors,
                                conf_hidden, ctypes.byref(out), workspace, workspace_bytes,
                                stream)


def dspark_prepare_head_size(cfg: dspark_config, head: dspark_head) -> int:
    return lib().dspark_prepare_head_size(ctypes.byref(cfg), ctypes.byref(head))


def dspark_prepare_head(cfg: dspark_config, head: dspark_head, prepared: int,
                        prepared_bytes: int, stream: int = 0) -> int:
    return lib().dspark_prepare_head(ctypes.byref(cfg), ctypes.byref(head), prepared,
                                     prepared_bytes, stream)


DSPARK_NUM_STAGES = 4
STAGE_NAMES = ("conf", "logits", "chain", "topk")


def dspark_propose_timed(cfg: dspark_config, head: dspark_head, hidden: int, anchors: int,
                         out: dspark_outputs, workspace: int, workspace_bytes: int,
                         stream: int, events, conf_hidden: int | None = None) -> int:
    """``events``: DSPARK_NUM_STAGES + 1 cudaEvent_t handles (ints)."""
    arr = (c_ptr * (DSPARK_NUM_STAGES + 1))(*events)
    return lib().dspark_propose_timed(ctypes.byref(cfg), ctypes.byref(head), hidden, anchors,
                                      conf_hidden, ctypes.byref(out), workspace,
                                      workspace_bytes, stream, arr)


def dspark_propose_kernel_count(cfg: dspark_config, head: dspark_head,
                                out: dspark_outputs) -> int:
    return lib().dspark_propose_kernel_count(ctypes.byref(cfg), ctypes.byref(head),
                                             ctypes.byref(out))


def dspark_step_host_workspace_size(cfg: dspark_config, head: dspark_head) -> int:
    return lib().dspark_step_host_workspace_size(ctypes.byref(cfg), ctypes.byref(head))


def dspark_step_host(cfg: dspark_config, head: dspark_head, hidden_h: int, anchors_h: int,
                     target_h: int, draft_h: int, n_draft_h: int, accepted_h: int,
                     bonus_h: int, topk_ids_h: int | None, topk_vals_h: int | None,
                     workspace: int, workspace_bytes: int, stream: int = 0,
                     conf_hidden_h: int | None = None) -> int:
    """``conf_hidden_h`` goes to the C argument of that name (after ``anchors_h``)."""
    return lib().dspark_step_host(ctypes.byref(cfg), ctypes.byref(head), hidden_h, anchors_h,
                                  conf_hidden_h, target_h, draft_h, n_draft_h, accepted_h,
                                  bonus_h, topk_ids_h, topk_vals_h, workspace, workspace_bytes,
                                  stream)


def dspark_propose_noalloc(cfg: dspark_config, head: dspark_head, hidden: int, anchors: int,
                           out: dspark_outputs, stream: int = 0,
                           conf_hidden: int | None = None) -> int:
    """dspark_propose with the library's built-in 16 MiB scratch (no workspace)."""
    return lib().dspark_propose_noalloc(ctypes.byref(cfg), ctypes.byref(head), hidden, anchors,
                                        conf_hidden, ctypes.byref(out), stream)


def dspark_verify(B: int, N: int, draft: int, n_draft: int, target: int, accepted: int,
                  bonus: int, emitted: int | None, stream: int = 0) -> int:
    return lib().dspark_verify(B, N, draft, n_draft, target, accepted, bonus, emitted,
                               stream)


def dspark_tree_verify(B: int, N: int, top_k: int, topk_ids: int, n_draft: int, target: int,
                       accepted: int, bonus: int, emitted: int | None, path: int | None,
                       stream: int = 0) -> int:
    return lib().dspark_tree_verify(B, N, top_k, topk_ids, n_draft, target, accepted, bonus,
                                    emitted, path, stream)


def dspark_device_status(workspace: int, stream: int = 0) -> int:
    return lib().dspark_device_status(workspace, stream)


def dspark_noalloc_device_status(stream: int = 0) -> int:
    return lib().dspark_noalloc_device_status(stream)


def dspark_pass_stats(workspace: int, stream: int = 0) -> dict:
    """Counters of the latest propose call on ``workspace`` (see include/dspark.h)."""
    a, b, c = c_i32(0), c_i32(0), c_i32(0)
    check(lib().dspark_pass_stats(workspace, stream, ctypes.byref(a), ctypes.byref(b),
                                  ctypes.byref(c)))
    return {"on_the_fly": a.value, "every_row": b.value, "dense_overflow": c.value}


def dspark_wait_selftest(workspace: int, workspace_bytes: int, budget_cycles: int,
                         pre_abort: bool = False, stream: int = 0) -> int:
    return lib().dspark_wait_selftest(workspace, workspace_bytes, budget_cycles,
                                      int(pre_abort), stream)


def dspark_status_string(status: int) -> str:
    return lib().dspark_status_string(status).decode()


def dspark_last_error() -> str:
    return lib().dspark_last_error().decode()
