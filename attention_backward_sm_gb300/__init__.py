"""Python binding of libfabwd.so: single-pass flash-attention backward on GB300.

The functions keep the C names of ``include/fabwd.h`` and only marshal
arguments (data pointers, sizes, the current CUDA stream).  Every step of
the computation runs in the library's CUDA kernels; PyTorch provides device
memory and streams.  ``backward`` chains the three backward calls and
allocates their outputs with torch.

Tensors: q, o, do, dq are [total_q, H, d] bf16; k, v, dk, dv are
[total_kv, Hkv, d] bf16 (Hkv divides H: grouped-query attention when it is
smaller); m, l, D are [total_q, H] float32; d is 64, 128 or 256; cu_q /
cu_kv are cumulative int32 offsets (B+1 entries) given both as a CUDA tensor
and as a host sequence.
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import _lib

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_TIMEOUT = 4
FA_DQ_ATOMIC = 0
FA_DQ_DETERMINISTIC = 1
FA_MASK_NONE = 0
FA_MASK_CAUSAL = 1
FA_MASK_CAUSAL_BOTTOM_RIGHT = 2


def mask_kind(causal: bool, bottom_right: bool = False) -> int:
    """fa_mask value for a causal flag and an alignment."""
    if not causal:
        if bottom_right:
            raise ValueError("bottom_right needs causal")
        return FA_MASK_NONE
    return FA_MASK_CAUSAL_BOTTOM_RIGHT if bottom_right else FA_MASK_CAUSAL


class FabwdError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"fabwd error {code}: {msg}")
        self.code = code


def lib():
    return _lib.load()


def fa_last_error() -> str:
    return (lib().fa_last_error() or b"").decode()


def _check(rc: int):
    if rc != FA_OK:
        raise FabwdError(rc, fa_last_error())


# The helpers below run on every call; they are kept to plain attribute
# reads because small problems are bound by the host time of a launch.
def _ptr(t) -> int | None:
    if t is None:
        return None
    return t.data_ptr() or None


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> int | None:
    if stream is not None:
        return stream.cuda_stream or None
    if _raw_stream is not None:
        return _raw_stream(torch.cuda.current_device()) or None
    return torch.cuda.current_stream().cuda_stream or None


def _host_offsets(cu) -> np.ndarray:
    if isinstance(cu, np.ndarray) and cu.dtype == np.int32 and cu.flags.c_contiguous:
        return cu
    if isinstance(cu, torch.Tensor):
        cu = cu.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(cu, dtype=np.int32))


def _hp(a: np.ndarray) -> int:
    return a.ctypes.data


def _shape(q):
    total, heads, dim = q.shape
    return int(total), int(heads), int(dim)


def fa_fwd_stats(q, k, v, o, m, l, cu_q_dev, cu_kv_dev, cu_q_host, cu_kv_host, causal: bool, scale: float,
                 stream=None):
    """Fills o (bf16), m and l (fp32) in place."""
    cq, ck = _host_offsets(cu_q_host), _host_offsets(cu_kv_host)
    total_q, heads, dim = _shape(q)
    total_kv = int(k.shape[0])
    _check(lib().fa_fwd_stats(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(m), _ptr(l), _ptr(cu_q_dev),
                              _ptr(cu_kv_dev), _hp(cq), _hp(ck), len(cq) - 1, total_q, total_kv, heads, dim,
                              int(bool(causal)), float(scale), _stream(stream)))


def fa_fwd_stats_gqa(q, k, v, o, m, l, cu_q_dev, cu_kv_dev, cu_q_host, cu_kv_host, causal: bool, scale: float,
                     stream=None):
    """fa_fwd_stats with k, v carrying k.shape[1] key/value heads."""
    cq, ck = _host_offsets(cu_q_host), _host_offsets(cu_kv_host)
    total_q, heads, dim = _shape(q)
    total_kv, heads_kv = int(k.shape[0]), int(k.shape[1])
    _check(lib().fa_fwd_stats_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(m), _ptr(l), _ptr(cu_q_dev),
                                  _ptr(cu_kv_dev), _hp(cq), _hp(ck), len(cq) - 1, total_q, total_kv, heads, heads_kv,
                                  dim, int(bool(causal)), float(scale), _stream(stream)))


def fa_fwd_stats_ex(q, k, v, o, m, l, cu_q_dev, cu_kv_dev, cu_q_host, cu_kv_host, mask: int, window: int,
                    scale: float, stream=None):
    """fa_fwd_stats_gqa with an fa_mask value and a sliding window (0 = none)."""
    cq, ck = _host_offsets(cu_q_host), _host_offsets(cu_kv_host)
    total_q, heads, dim = _shape(q)
    total_kv, heads_kv = int(k.shape[0]), int(k.shape[1])
    _check(lib().fa_fwd_stats_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(m), _ptr(l), _ptr(cu_q_dev),
                                 _ptr(cu_kv_dev), _hp(cq), _hp(ck), len(cq) - 1, total_q, total_kv, heads, heads_kv,
                                 dim, int(mask), int(window), float(scale), _stream(stream)))


def fa_fwd_lse(q, k, v, o, lse, cu_q_dev, cu_kv_dev, cu_q_host, cu_kv_host, mask: int, window: int, scale: float,
               stream=None):
    """fa_fwd_stats_ex writing lse = m + ln(l) per row instead of (m, l)."""
    cq, ck = _host_offsets(cu_q_host), _host_offsets(cu_kv_host)
    total_q, heads, dim = _shape(q)
    total_kv, heads_kv = int(k.shape[0]), int(k.shape[1])
    _check(lib().fa_fwd_lse(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_q_dev), _ptr(cu_kv_dev), _hp(cq),
                            _hp(ck), len(cq) - 1, total_q, total_kv, heads, heads_kv, dim, int(mask), int(window),
                            float(scale), _stream(stream)))


def fa_bwd_preprocess(o, do, D, dq_acc, stream=None):
    total_q, heads, dim = _shape(o)
    _check(lib().fa_bwd_preprocess(_ptr(o), _ptr(do), _ptr(D), _ptr(dq_acc), total_q, heads, dim,
                                   _stream(stream)))


def fa_bwd_workspace_size(cu_q_host, cu_kv_host, heads: int, head_dim: int, causal: bool, dq_mode: int) -> int:
    cq, ck = _host_offsets(cu_q_host), _host_offsets(cu_kv_host)
    n = lib().fa_bwd_workspace_size(_hp(cq), _hp(ck), len(cq) - 1, heads, head_dim, int(bool(causal)), dq_mode)
    err = fa_last_error()
    if err:
        raise FabwdError(FA_ERR_INVALID_ARG, err)
    return int(n)


def fa_bwd(q, k, v, do, m, l, D, dq_acc, dk, dv, cu_q_dev, cu_kv_dev, cu_q_host, cu_kv_host, causal: bool,
           scale: float, dq_mode: int = FA_DQ_ATOMIC, workspace=None, stream=None):
    cq, ck = _host_offsets(cu_q_host), _host_offsets(cu_kv_host)
    total_q, heads, dim = _shape(q)
    total_kv = int(k.shape[0])
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(m), _ptr(l), _ptr(D), _ptr(dq_acc), _ptr(dk),
                        _ptr(dv), _ptr(cu_q_dev), _ptr(cu_kv_dev), _hp(cq), _hp(ck), len(cq) - 1, total_q, total_kv,
                        heads, dim, int(bool(causal)), float(scale), int(dq_mode), _ptr(workspace), ws_bytes,
                        _stream(stream)))


def fa_bwd_gqa(q, k, v, do, m, l, D, dq_acc, dk, dv, cu_q_dev, cu_kv_dev, cu_q_host, cu_kv_host, causal: bool,
               scale: float, dq_mode: int = FA_DQ_ATOMIC, workspace=None, stream=None):
    """fa_bwd with k, v, dk, dv carrying k.shape[1] key/value heads."""
    cq, ck = _host_offsets(cu_q_host), _host_offsets(cu_kv_host)
    total_q, heads, dim = _shape(q)
    total_kv, heads_kv = int(k.shape[0]), int(k.shape[1])
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().fa_bwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(m), _ptr(l), _ptr(D), _ptr(dq_acc),
                            _ptr(dk), _ptr(dv), _ptr(cu_q_dev), _ptr(cu_kv_dev), _hp(cq), _hp(ck), len(cq) - 1,
                            total_q, total_kv, heads, heads_kv, dim, int(bool(causal)), float(scale), int(dq_mode),
                            _ptr(workspace), ws_bytes, _stream(stream)))


def fa_bwd_ex(q, k, v, do, m, l, D, dq_acc, dk, dv, cu_q_dev, cu_kv_dev, cu_q_host, cu_kv_host, mask: int,
              window: int, scale: float, dq_mode: int = FA_DQ_ATOMIC, workspace=None, stream=None):
    """fa_bwd_gqa with an fa_mask value and a sliding window (0 = none)."""
    cq, ck = _host_offsets(cu_q_host), _host_offsets(cu_kv_host)
    total_q, heads, dim = _shape(q)
    total_kv, heads_kv = int(k.shape[0]), int(k.shape[1])
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().fa_bwd_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(m), _ptr(l), _ptr(D), _ptr(dq_acc),
                           _ptr(dk), _ptr(dv), _ptr(cu_q_dev), _ptr(cu_kv_dev), _hp(cq), _hp(ck), len(cq) - 1,
                           total_q, total_kv, heads, heads_kv, dim, int(mask), int(window), float(scale),
                           int(dq_mode), _ptr(workspace), ws_bytes, _stream(stream)))


def fa_bwd_lse(q, k, v, do, lse, D, dq_acc, dk, dv, cu_q_dev, cu_kv_dev, cu_q_host, cu_kv_host, mask: int,
               window: int, scale: float, dq_mode: int = FA_DQ_ATOMIC, workspace=None, stream=None):
    """fa_bwd_ex from the single statistic lse instead of (m, l)."""
    cq, ck = _host_offsets(cu_q_host), _host_offsets(cu_kv_host)
    total_q, heads, dim = _shape(q)
    total_kv, heads_kv = int(k.shape[0]), int(k.shape[1])
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().fa_bwd_lse(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(lse), _ptr(D), _ptr(dq_acc), _ptr(dk),
                            _ptr(dv), _ptr(cu_q_dev), _ptr(cu_kv_dev), _hp(cq), _hp(ck), len(cq) - 1, total_q,
                            total_kv, heads, heads_kv, dim, int(mask), int(window), float(scale), int(dq_mode),
                            _ptr(workspace), ws_bytes, _stream(stream)))


def fa_bwd_dq_finalize(dq_acc, dq, scale: float, stream=None):
    total_q, heads, dim = _shape(dq)
    _check(lib().fa_bwd_dq_finalize(_ptr(dq_acc), _ptr(dq), total_q, heads, dim, float(scale), _stream(stream)))


def fa_bwd_noalloc(q, k, v, o, do, m, l, dq, dk, dv, cu_q_dev, cu_kv_dev, cu_q_host, cu_kv_host, causal: bool,
                   scale: float, stream=None):
    """Whole backward into caller-provided dq, dk, dv with the library's own
    fixed scratch array (no device allocation anywhere on the call)."""
    cq, ck = _host_offsets(cu_q_host), _host_offsets(cu_kv_host)
    total_q, heads, dim = _shape(q)
    total_kv = int(k.shape[0])
    _check(lib().fa_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(m), _ptr(l), _ptr(dq), _ptr(dk),
                                _ptr(dv), _ptr(cu_q_dev), _ptr(cu_kv_dev), _hp(cq), _hp(ck), len(cq) - 1, total_q,
                                total_kv, heads, dim, int(bool(causal)), float(scale), _stream(stream)))


def fa_selftest_wait_timeout(stream=None):
    """Launches a block whose bounded wait runs out (after 1 s); the next
    fa_check_device_status raises FabwdError with FA_ERR_TIMEOUT."""
    _check(lib().fa_selftest_wait_timeout(_stream(stream)))


def fa_check_device_status(stream=None):
    _check(lib().fa_check_device_status(_stream(stream)))


def forward_stats(q, k, v, cu_q_dev, cu_kv_dev, cu_q_host, cu_kv_host, causal: bool, scale: float, stream=None,
                  window: int = 0, bottom_right: bool = False, check: bool = True):
    """Allocates and returns (o, m, l) from fa_fwd_stats_ex (k, v may have
    fewer heads than q; window > 0 is a causal sliding window).  check:
    wait for the stream and raise unless the device status word is clean
    (a kernel whose bounded wait ran out leaves partial outputs)."""
    total_q, heads, dim = _shape(q)
    o = torch.zeros_like(q)
    m = torch.zeros((total_q, heads), dtype=torch.float32, device=q.device)
    l = torch.zeros((total_q, heads), dtype=torch.float32, device=q.device)
    fa_fwd_stats_ex(q, k, v, o, m, l, cu_q_dev, cu_kv_dev, cu_q_host, cu_kv_host, mask_kind(causal, bottom_right),
                    window, scale, stream)
    if check:
        fa_check_device_status(stream)
    return o, m, l


class Workspace:
    """Device buffers one backward needs besides its inputs and outputs."""

    def __init__(self, q, cu_q_host, cu_kv_host, causal, dq_mode):
        total_q, heads, dim = _shape(q)
        self.D = torch.empty((total_q, heads), dtype=torch.float32, device=q.device)
        self.dq_acc = torch.empty((total_q, heads, dim), dtype=torch.float32, device=q.device)
        n = fa_bwd_workspace_size(cu_q_host, cu_kv_host, heads, dim, causal, dq_mode)
        self.ws = torch.empty(max(n, 1), dtype=torch.uint8, device=q.device) if n > 0 else None


def backward(q, k, v, o, do, m, l, cu_q_dev, cu_kv_dev, cu_q_host, cu_kv_host, causal: bool, scale: float,
             dq_mode: int = FA_DQ_ATOMIC, out=None, work: Workspace | None = None, stream=None,
             window: int = 0, bottom_right: bool = False, check: bool = True):
    """preprocess -> fa_bwd_ex -> finalize on one stream; returns (dq, dk, dv).
    k and v may have fewer heads than q (grouped-query attention); the mask
    is none, causal (top-left, or bottom-right) and optionally a causal
    sliding window of `window` keys.  check (default): wait for the stream
    and raise FabwdError unless the device status word is clean, so that
    gradients left partial by a timed-out wait are never returned; pass
    check=False to keep the call asynchronous and call
    fa_check_device_status() before using the results."""
    if work is None:
        work = Workspace(q, cu_q_host, cu_kv_host, causal, dq_mode)
    if out is None:
        out = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    dq, dk, dv = out
    fa_bwd_preprocess(o, do, work.D, work.dq_acc, stream)
    fa_bwd_ex(q, k, v, do, m, l, work.D, work.dq_acc, dk, dv, cu_q_dev, cu_kv_dev, cu_q_host, cu_kv_host,
              mask_kind(causal, bottom_right), window, scale, dq_mode, work.ws, stream)
    fa_bwd_dq_finalize(work.dq_acc, dq, scale, stream)
    if check:
        fa_check_device_status(stream)
    return dq, dk, dv


def forward_lse(q, k, v, cu_q_dev, cu_kv_dev, cu_q_host, cu_kv_host, causal: bool, scale: float, stream=None,
                window: int = 0, bottom_right: bool = False, check: bool = True):
    """Allocates and returns (o, lse) from fa_fwd_lse (check: as in
    forward_stats)."""
    total_q, heads, dim = _shape(q)
    o = torch.zeros_like(q)
    lse = torch.zeros((total_q, heads), dtype=torch.float32, device=q.device)
    fa_fwd_lse(q, k, v, o, lse, cu_q_dev, cu_kv_dev, cu_q_host, cu_kv_host, mask_kind(causal, bottom_right), window,
               scale, stream)
    if check:
        fa_check_device_status(stream)
    return o, lse


def backward_lse(q, k, v, o, do, lse, cu_q_dev, cu_kv_dev, cu_q_host, cu_kv_host, causal: bool, scale: float,
                 dq_mode: int = FA_DQ_ATOMIC, out=None, work: Workspace | None = None, stream=None,
                 window: int = 0, bottom_right: bool = False, check: bool = True):
    """backward() from the single statistic lse = m + ln(l) (check: as in
    backward)."""
    if work is None:
        work = Workspace(q, cu_q_host, cu_kv_host, causal, dq_mode)
    if out is None:
        out = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    dq, dk, dv = out
    fa_bwd_preprocess(o, do, work.D, work.dq_acc, stream)
    fa_bwd_lse(q, k, v, do, lse, work.D, work.dq_acc, dk, dv, cu_q_dev, cu_kv_dev, cu_q_host, cu_kv_host,
               mask_kind(causal, bottom_right), window, scale, dq_mode, work.ws, stream)
    fa_bwd_dq_finalize(work.dq_acc, dq, scale, stream)
    if check:
        fa_check_device_status(stream)
    return dq, dk, dv
