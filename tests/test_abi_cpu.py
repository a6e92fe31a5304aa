"""The C-ABI library without a GPU: it loads, exports every declared symbol, and its
host-side validation answers with status codes before touching the device."""
import ctypes
import os
import re

import pytest

import dspark_block_drafter_gb300 as ds
from dspark_block_drafter_gb300 import _abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^[A-Za-z_][\w \*]*?\b(dspark_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_abi.LIB_PATH):
        from dspark_block_drafter_gb300 import build
        build.build()
    return ds.lib()


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert "dspark_propose" in names and "dspark_verify" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
        assert n in _abi.SIGNATURES, f"{n} has no Python binding"


def _cfg(**kw):
    c = dict(B=2, L_in=4, H=64, V=1000, r=8, top_k=4, sample_from_anchor=1, topk_markov=1,
             conf_min=0.0, dtype=_abi.DSPARK_F32)
    c.update(kw)
    return _abi.dspark_config(**c)


def _head(**kw):
    h = dict(lm_head=0x1000, lm_bias=None, d2t=None, V_head=1000, markov_w1=0x2000,
             markov_w2=0x3000, w_conf=None, b_conf=0.0)
    h.update(kw)
    return _abi.dspark_head(**h)


def test_num_slots(lib):
    assert ds.dspark_num_slots(_cfg(L_in=7, sample_from_anchor=1)) == 7
    assert ds.dspark_num_slots(_cfg(L_in=7, sample_from_anchor=0)) == 6
    assert ds.dspark_num_slots(_cfg(L_in=1, sample_from_anchor=0)) == 0


def test_workspace_size_and_validation(lib):
    n = ds.dspark_propose_workspace_size(_cfg(), _head())
    assert n > 0 and n % 256 == 0
    # the workspace holds at least the fp32 base logits of every prediction slot
    assert n >= 4 * 2 * 4 * 1000
    bad = [
        _cfg(B=0), _cfg(top_k=0), _cfg(top_k=33), _cfg(L_in=1, sample_from_anchor=0),
        _cfg(dtype=7), _cfg(sample_from_anchor=2), _cfg(conf_min=float("nan")),
    ]
    for c in bad:
        assert ds.dspark_propose_workspace_size(c, _head()) == 0
    assert ds.dspark_propose_workspace_size(_cfg(), _head(V_head=999)) == 0   # no d2t
    assert ds.dspark_propose_workspace_size(_cfg(), _head(lm_head=None)) == 0
    assert ds.dspark_propose_workspace_size(_cfg(top_k=5), _head(V_head=4, d2t=0x10)) == 0
    # bf16 alignment / size rules
    assert ds.dspark_propose_workspace_size(_cfg(dtype=1, H=60), _head()) == 0
    assert ds.dspark_propose_workspace_size(_cfg(dtype=1), _head(lm_head=0x1002)) == 0
    assert ds.dspark_propose_workspace_size(_cfg(dtype=1), _head()) > 0
    # the bf16 path takes at most 256 prediction slots and a Markov rank of at most 512
    assert ds.dspark_propose_workspace_size(_cfg(dtype=1, L_in=256), _head()) > 0
    assert ds.dspark_propose_workspace_size(_cfg(dtype=1, L_in=257), _head()) == 0
    assert ds.dspark_propose_workspace_size(_cfg(dtype=1, L_in=257, sample_from_anchor=0),
                                            _head()) > 0
    assert ds.dspark_propose_workspace_size(_cfg(dtype=1, r=512), _head()) > 0
    assert ds.dspark_propose_workspace_size(_cfg(dtype=1, r=520), _head()) == 0


def test_propose_rejects_before_launch(lib):
    out = _abi.dspark_outputs(draft=0x100, n_draft=0x200)
    cfg, head = _cfg(), _head()
    need = ds.dspark_propose_workspace_size(cfg, head)
    st = ds.dspark_propose(cfg, head, 0x4000, 0x5000, out, 0x10000, need - 1, 0)
    assert st == _abi.DSPARK_ERR_WORKSPACE
    assert "too small" in ds.dspark_last_error()
    st = ds.dspark_propose(cfg, head, 0x4000, 0x5000, out, 0x10010, need, 0)
    assert st == _abi.DSPARK_ERR_WORKSPACE                      # misaligned
    st = ds.dspark_propose(cfg, head, None, 0x5000, out, 0x10000, need, 0)
    assert st == _abi.DSPARK_ERR_INVALID_ARG
    st = ds.dspark_propose(cfg, head, 0x4000, 0x5000, _abi.dspark_outputs(draft=0x100),
                           0x10000, need, 0)
    assert st == _abi.DSPARK_ERR_INVALID_ARG
    st = ds.dspark_propose(_cfg(B=-1), head, 0x4000, 0x5000, out, 0x10000, need, 0)
    assert st == _abi.DSPARK_ERR_INVALID_ARG


def test_verify_rejects_before_launch(lib):
    assert ds.dspark_verify(0, 4, 1, 1, 1, 1, 1, None, 0) == _abi.DSPARK_ERR_INVALID_ARG
    assert ds.dspark_verify(2, 4, None, 1, 1, 1, 1, None, 0) == _abi.DSPARK_ERR_INVALID_ARG


def test_status_strings(lib):
    for s in range(7):
        assert ds.dspark_status_string(s)
    assert ds.dspark_status_string(99) == "unknown status"


def test_struct_layouts_match_c():
    # pointer-sized fields are 8 bytes on both hosts; the int/float fields pack as in C
    assert ctypes.sizeof(_abi.dspark_config) == 44
    assert ctypes.sizeof(_abi.dspark_head) == 72
    assert ctypes.sizeof(_abi.dspark_outputs) == 48


def test_skip_truncated_checked_before_launch(lib):
    head = _head()
    # not 0/1: invalid configuration, no workspace size
    assert ds.dspark_propose_workspace_size(_cfg(dtype=1, skip_truncated=2), head) == 0
    # the fp32 path has no adaptive form: refused before any launch
    cfg = _cfg(skip_truncated=1)
    need = ds.dspark_propose_workspace_size(cfg, head)
    assert need > 0
    out = _abi.dspark_outputs(draft=0x100, n_draft=0x200)
    st = ds.dspark_propose(cfg, head, 0x4000, 0x5000, out, 0x10000, need, 0)
    assert st == _abi.DSPARK_ERR_UNSUPPORTED


def test_wait_selftest_checked_before_launch(lib):
    # every refusal comes before a launch, so none of these needs a GPU
    W = _abi.DSPARK_ERR_WORKSPACE
    I = _abi.DSPARK_ERR_INVALID_ARG
    assert ds.dspark_wait_selftest(None, 256, 1000) == W
    assert ds.dspark_wait_selftest(0x10010, 256, 1000) == W          # not 256-byte aligned
    assert ds.dspark_wait_selftest(0x10000, 255, 1000) == W
    assert ds.dspark_wait_selftest(0x10000, 256, 0) == I
    assert ds.dspark_wait_selftest(0x10000, 256, 2_000_000_001) == I
    assert ds.dspark_wait_selftest(0x10000, 256, 1000, pre_abort=2) == I


def test_step_host_checked_before_launch(lib):
    cfg, head = _cfg(), _head()
    need = ds._abi.dspark_step_host_workspace_size(cfg, head)
    # the staging area comes on top of the proposal's workspace
    assert need > ds.dspark_propose_workspace_size(cfg, head)
    assert ds._abi.dspark_step_host_workspace_size(_cfg(B=0), head) == 0
    bufs = [0x1000 * (i + 1) for i in range(7)]          # hidden .. bonus (host)
    for i in range(7):                                   # each required buffer
        b = list(bufs)
        b[i] = None
        st = ds._abi.dspark_step_host(cfg, head, *b, None, None, 0x100000, need, 0)
        assert st == _abi.DSPARK_ERR_INVALID_ARG, i
    st = ds._abi.dspark_step_host(cfg, head, *bufs, None, None, 0x100000, need - 1, 0)
    assert st == _abi.DSPARK_ERR_WORKSPACE
    st = ds._abi.dspark_step_host(cfg, head, *bufs, None, None, 0x100010, need, 0)
    assert st == _abi.DSPARK_ERR_WORKSPACE


def test_prepare_head_checked_before_launch(lib):
    bf16 = _cfg(dtype=1)
    head = _head()
    need = ds._abi.dspark_prepare_head_size(bf16, head)
    assert need > 0 and need % 256 == 0
    # the prepared head holds markov_w2 transposed (bf16, padded rows), column norms etc.
    assert need >= 2 * 8 * 1000
    assert ds._abi.dspark_prepare_head_size(_cfg(), head) == 0          # fp32: not used
    assert ds._abi.dspark_prepare_head(_cfg(), head, 0x100000, need, 0) == \
        _abi.DSPARK_ERR_UNSUPPORTED
    assert ds._abi.dspark_prepare_head(bf16, head, None, need, 0) == _abi.DSPARK_ERR_WORKSPACE
    assert ds._abi.dspark_prepare_head(bf16, head, 0x100010, need, 0) == \
        _abi.DSPARK_ERR_WORKSPACE
    assert ds._abi.dspark_prepare_head(bf16, head, 0x100000, need - 1, 0) == \
        _abi.DSPARK_ERR_WORKSPACE
    assert ds._abi.dspark_prepare_head(_cfg(dtype=1, B=0), head, 0x100000, need, 0) == \
        _abi.DSPARK_ERR_INVALID_ARG


def test_timed_and_kernel_count_checked(lib):
    cfg, head = _cfg(), _head()
    out = _abi.dspark_outputs(draft=0x100, n_draft=0x200)
    need = ds.dspark_propose_workspace_size(cfg, head)
    n = _abi.DSPARK_NUM_STAGES + 1
    st = ds._abi.dspark_propose_timed(cfg, head, 0x4000, 0x5000, out, 0x10000, need, 0,
                                      [0x10] * (n - 1) + [None])
    assert st == _abi.DSPARK_ERR_INVALID_ARG                # an event is NULL
    st = ds._abi.dspark_propose_timed(cfg, head, 0x4000, 0x5000, out, 0x10000, need - 1, 0,
                                      [0x10] * n)
    assert st == _abi.DSPARK_ERR_WORKSPACE
    # launches per pass (each starts with the control-block reset) on the fp32 path:
    # confidence, GEMM and the one-launch chain; or, when a GPU says this small shape
    # fits, the chain alone (it evaluates both)
    assert ds._abi.dspark_propose_kernel_count(cfg, head, out) in (2, 4)
    # bf16, no prepared head: reset, confidence, GEMM, one chain launch per 32 blocks,
    # top-k
    bf = _cfg(dtype=1, B=70)
    topk = _abi.dspark_outputs(draft=0x100, n_draft=0x200, topk_ids=0x300, topk_vals=0x400)
    assert ds._abi.dspark_propose_kernel_count(bf, head, topk) == 1 + 1 + 1 + 3 + 1
    assert ds._abi.dspark_propose_kernel_count(bf, head, out) == 1 + 1 + 1 + 3
    # a prepared head: reset, the GEMM and the tables with the walk; the confidence kernel
    # before the GEMM when the block length is adaptive
    prep = _head(prepared=0x9000)
    assert ds._abi.dspark_propose_kernel_count(bf, prep, topk) == 3
    assert ds._abi.dspark_propose_kernel_count(_cfg(dtype=1, B=70, skip_truncated=1), prep,
                                               topk) == 4
    assert ds._abi.dspark_propose_kernel_count(_cfg(B=0), head, out) == -1


def test_noalloc_checked_before_launch(lib):
    out = _abi.dspark_outputs(draft=0x100, n_draft=0x200)
    # an invalid configuration answers as dspark_propose would
    st = ds._abi.dspark_propose_noalloc(_cfg(B=0), _head(), 0x4000, 0x5000, out, 0)
    assert st == _abi.DSPARK_ERR_INVALID_ARG
    # a call whose scratch would exceed 16 MiB is refused on the host
    big = _cfg(B=64, L_in=16, V=100000)
    st = ds._abi.dspark_propose_noalloc(big, _head(V_head=100000), 0x4000, 0x5000, out, 0)
    assert st == _abi.DSPARK_ERR_WORKSPACE
    assert "16777216" in ds.dspark_last_error()


def test_header_is_plain_c():
    # the boundary is a C ABI: the header must compile as strict C99 with no CUDA or C++
    # types, and a C caller must be able to name every entry point (source through stdin,
    # object to /dev/null: nothing is written)
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    names = _declared_functions()
    src = ['#include "dspark.h"', "typedef void (*any_fn)(void);", "int main(void) {",
           "  dspark_config c = {0}; dspark_head h = {0}; dspark_outputs o = {0};",
           "  any_fn f;", "  (void)c; (void)h; (void)o;"]
    src += [f"  f = (any_fn)&{n}; (void)f;" for n in names]
    src += ["  return DSPARK_OK + DSPARK_NUM_STAGES * 0;", "}"]
    r = subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        "-I", os.path.join(ROOT, "include"), "-x", "c", "-c", "-",
                        "-o", os.devnull], input="\n".join(src) + "\n",
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_pass_stats_refuses_null_workspace(lib):
    import ctypes
    a = ctypes.c_int32(0)
    assert lib.dspark_pass_stats(None, None, ctypes.byref(a), None, None) == \
        _abi.DSPARK_ERR_INVALID_ARG
