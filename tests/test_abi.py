"""The C-ABI library builds, loads without a GPU and exports every entry
point declared in include/fabwd.h; host-side argument checks return their
error codes before anything touches the device."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "fabwd.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from attention_backward_sm_gb300 import build
    build.build()
    from attention_backward_sm_gb300 import _lib
    return _lib.load()


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ("fa_fwd_stats", "fa_fwd_stats_gqa", "fa_bwd_preprocess", "fa_bwd", "fa_bwd_gqa",
                 "fa_bwd_dq_finalize", "fa_bwd_workspace_size",
                 "fa_check_device_status", "fa_last_error"):
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    from attention_backward_sm_gb300 import _lib
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"binding lacks {name}"


def _offsets(*xs):
    return np.asarray(xs, dtype=np.int32)


def _call_bwd(lib, cu_q, cu_kv, heads=2, head_dim=128, causal=0, dq_mode=0, total_q=None, total_kv=None,
              scale=0.1):
    p = ctypes.c_void_p(16)   # never dereferenced: the checks fail first
    total_q = int(cu_q[-1]) if total_q is None else total_q
    total_kv = int(cu_kv[-1]) if total_kv is None else total_kv
    return lib.fa_bwd(p, p, p, p, p, p, p, p, p, p, p, p, cu_q.ctypes.data_as(ctypes.c_void_p),
                      cu_kv.ctypes.data_as(ctypes.c_void_p), len(cu_q) - 1, total_q, total_kv, heads, head_dim,
                      causal, scale, dq_mode, None, 0, None)


def test_host_argument_checks(lib):
    cu = _offsets(0, 10, 30)
    assert _call_bwd(lib, cu, cu, head_dim=96) == 2            # FA_ERR_UNSUPPORTED
    assert b"head_dim" in lib.fa_last_error()
    assert _call_bwd(lib, _offsets(0, 10, 5), cu) == 1         # decreasing offsets
    assert b"non-decreasing" in lib.fa_last_error()
    assert _call_bwd(lib, _offsets(1, 10, 30), cu) == 1        # cu[0] != 0
    assert _call_bwd(lib, cu, cu, total_kv=20) == 1            # offsets exceed the tensor
    assert _call_bwd(lib, cu, cu, heads=0) == 1
    assert _call_bwd(lib, cu, cu, causal=2) == 1
    assert _call_bwd(lib, cu, cu, dq_mode=7) == 1
    assert _call_bwd(lib, cu, cu, scale=float("inf")) == 1
    p = ctypes.c_void_p(16)
    assert lib.fa_bwd_preprocess(p, p, p, p, 10, 2, 80, None) == 2
    assert lib.fa_bwd_dq_finalize(p, p, 10, 0, 128, 1.0, None) == 1
    # an empty problem is a successful no-op
    z = _offsets(0)
    assert _call_bwd(lib, z, z, total_q=0, total_kv=0) == 0
    assert lib.fa_last_error() == b""


def test_workspace_size(lib):
    cu = _offsets(0, 300, 700)
    hp = cu.ctypes.data_as(ctypes.c_void_p)
    assert lib.fa_bwd_workspace_size(hp, hp, 2, 4, 128, 1, 0) == 0
    # deterministic at head_dim 64 / 128: dQ is summed per row by one CTA, no counters
    assert lib.fa_bwd_workspace_size(hp, hp, 2, 4, 128, 1, 1) == 0
    assert lib.fa_bwd_workspace_size(hp, hp, 2, 4, 64, 0, 1) == 0
    assert lib.fa_bwd_workspace_size(hp, hp, 2, 4, 128, 1, 5) == 0
    assert b"dq_mode" in lib.fa_last_error()


def test_gqa_host_argument_checks(lib):
    """fa_bwd_gqa / fa_fwd_stats_gqa reject head counts that do not form
    equal groups before touching the device."""
    cu = _offsets(0, 10, 30)
    hp = cu.ctypes.data_as(ctypes.c_void_p)
    p = ctypes.c_void_p(16)
    for heads, heads_kv in ((6, 4), (4, 0), (4, -2), (2, 4)):
        rc = lib.fa_bwd_gqa(p, p, p, p, p, p, p, p, p, p, p, p, hp, hp, 2, 30, 30, heads, heads_kv, 128, 0, 0.1, 0,
                            None, 0, None)
        assert rc == 1, (heads, heads_kv)
        assert b"multiple" in lib.fa_last_error()
        rc = lib.fa_fwd_stats_gqa(p, p, p, p, p, p, p, p, hp, hp, 2, 30, 30, heads, heads_kv, 128, 0, 0.1, None)
        assert rc == 1, (heads, heads_kv)
    # shape checks still come first
    assert lib.fa_bwd_gqa(p, p, p, p, p, p, p, p, p, p, p, p, hp, hp, 2, 30, 30, 4, 2, 96, 0, 0.1, 0,
                          None, 0, None) == 2


def _call_bwd_ex(lib, cu_q, cu_kv, mask=1, window=0, heads=2, heads_kv=2, head_dim=128, dq_mode=0):
    p = ctypes.c_void_p(16)
    hq, hk = cu_q.ctypes.data_as(ctypes.c_void_p), cu_kv.ctypes.data_as(ctypes.c_void_p)
    return lib.fa_bwd_ex(p, p, p, p, p, p, p, p, p, p, p, p, hq, hk, len(cu_q) - 1, int(cu_q[-1]), int(cu_kv[-1]),
                         heads, heads_kv, head_dim, mask, window, 0.1, dq_mode, None, 0, None)


def test_mask_and_window_argument_checks(lib):
    """fa_bwd_ex / fa_fwd_stats_ex reject unknown masks, negative windows and
    a window without a causal mask before touching the device."""
    cu = _offsets(0, 10, 30)
    assert _call_bwd_ex(lib, cu, cu, mask=3) == 1
    assert b"mask" in lib.fa_last_error()
    assert _call_bwd_ex(lib, cu, cu, mask=-1) == 1
    assert _call_bwd_ex(lib, cu, cu, mask=1, window=-5) == 1
    assert b"window" in lib.fa_last_error()
    assert _call_bwd_ex(lib, cu, cu, mask=0, window=4) == 1
    assert b"causal" in lib.fa_last_error()
    p = ctypes.c_void_p(16)
    hp = cu.ctypes.data_as(ctypes.c_void_p)
    assert lib.fa_fwd_stats_ex(p, p, p, p, p, p, p, p, hp, hp, 2, 30, 30, 2, 2, 128, 0, 7, 0.1, None) == 1
    assert lib.fa_fwd_lse(p, p, p, p, p, p, p, hp, hp, 2, 30, 30, 2, 2, 128, 5, 0, 0.1, None) == 1
    # the plain entry points keep accepting only a 0/1 causal flag
    assert _call_bwd(lib, cu, cu, causal=2) == 1


def test_head_dim_256_is_accepted_and_others_are_not(lib):
    cu = _offsets(0, 10, 30)
    # head_dim 256 passes the shape checks (then stops at a NULL device pointer, not UNSUPPORTED)
    p = ctypes.c_void_p(16)
    hp = cu.ctypes.data_as(ctypes.c_void_p)
    rc = lib.fa_bwd_ex(None, None, None, None, None, None, None, None, None, None, None, None, hp, hp, 2, 30, 30,
                       2, 2, 256, 1, 0, 0.1, 0, None, 0, None)
    assert rc == 1 and b"NULL" in lib.fa_last_error()
    for d in (32, 96, 192, 512):
        assert _call_bwd_ex(lib, cu, cu, head_dim=d) == 2
        assert b"head_dim" in lib.fa_last_error()
    assert lib.fa_bwd_preprocess(p, p, p, p, 10, 2, 192, None) == 2


def test_workspace_size_head_dim_256(lib):
    """Deterministic mode at head_dim 256 counts 64-row query blocks, two
    head-dim halves and four 32-dim quarters per (batch, head)."""
    cu = _offsets(0, 300, 700)
    hp = cu.ctypes.data_as(ctypes.c_void_p)
    n = lib.fa_bwd_workspace_size(hp, hp, 2, 4, 256, 0, 1)
    assert n >= 2 * 4 * 7 * 8 * 4 and n % 256 == 0            # max_q = 400 -> 7 blocks of 64
    assert lib.fa_bwd_workspace_size(hp, hp, 2, 4, 256, 0, 0) == 0


def test_lse_entry_points_need_no_l(lib):
    """fa_bwd_lse has no l argument: with no work it succeeds, and its
    pointer checks do not ask for one."""
    z = _offsets(0)
    hp = z.ctypes.data_as(ctypes.c_void_p)
    assert lib.fa_bwd_lse(None, None, None, None, None, None, None, None, None, None, None, hp, hp, 0, 0, 0,
                          2, 2, 128, 1, 0, 0.1, 0, None, 0, None) == 0


def _call_noalloc(lib, cu_q, cu_kv, heads=2, head_dim=128, causal=0, total_q=None, total_kv=None, scale=0.1,
                  ptr=16):
    p = ctypes.c_void_p(ptr)   # never dereferenced: the checks fail first
    total_q = int(cu_q[-1]) if total_q is None else total_q
    total_kv = int(cu_kv[-1]) if total_kv is None else total_kv
    return lib.fa_bwd_noalloc(p, p, p, p, p, p, p, p, p, p, p, p, cu_q.ctypes.data_as(ctypes.c_void_p),
                              cu_kv.ctypes.data_as(ctypes.c_void_p), len(cu_q) - 1, total_q, total_kv, heads,
                              head_dim, causal, scale, None)


def test_noalloc_checks_every_argument_before_any_cuda_call(lib):
    """fa_bwd_noalloc rejects bad arguments with the same codes as fa_bwd
    before it touches CUDA at all (here there is no GPU, so any CUDA call
    would turn into FA_ERR_CUDA instead)."""
    good = _offsets(0, 10, 30)
    assert _call_noalloc(lib, _offsets(0, 40, 30), good, total_q=40) == 1    # decreasing offsets
    assert b"non-decreasing" in lib.fa_last_error()
    assert _call_noalloc(lib, _offsets(1, 10, 30), good) == 1                # cu[0] != 0
    assert _call_noalloc(lib, good, _offsets(0, 10, 50), total_kv=30) == 1   # offsets past the tensor
    assert _call_noalloc(lib, good, good, head_dim=96) == 2                  # FA_ERR_UNSUPPORTED
    assert _call_noalloc(lib, good, good, causal=2) == 1
    assert _call_noalloc(lib, good, good, scale=float("nan")) == 1
    assert _call_noalloc(lib, good, good, ptr=8) == 1                        # misaligned pointers
    assert b"aligned" in lib.fa_last_error()
    # too large for the fixed array: total_q * heads * (head_dim + 1) * 4 > 16 MiB
    big = _offsets(0, 40000)
    assert _call_noalloc(lib, big, _offsets(0, 8), heads=8, head_dim=256) == 1
    assert b"scratch" in lib.fa_last_error()
    # head_dim 256 passes the shape checks: it then stops at a NULL device
    # pointer (INVALID_ARG), not at the head dimension (UNSUPPORTED)
    p = ctypes.c_void_p(16)
    hp = good.ctypes.data_as(ctypes.c_void_p)
    rc = lib.fa_bwd_noalloc(None, p, p, p, p, p, p, p, p, p, p, p, hp, hp, 2, 30, 30, 2, 256, 0, 0.1, None)
    assert rc == 1 and b"NULL" in lib.fa_last_error()
