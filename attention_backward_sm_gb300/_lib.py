"""ctypes loader for libfabwd.so (built in-tree by ``build.py``).

There is no fallback: if the library is missing or fails to load, importing
the binding raises, so a GPU run can never silently take another path.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfabwd.so")

# name -> (restype, argtypes), mirroring include/fabwd.h
_p = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t
SIGNATURES = {
    "fa_fwd_stats": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _f, _p]),
    "fa_fwd_stats_gqa": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _f, _p]),
    "fa_fwd_stats_ex": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _f, _p]),
    "fa_fwd_lse": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _i, _i, _f, _p]),
    "fa_bwd_preprocess": (_i, [_p, _p, _p, _p, _i, _i, _i, _p]),
    "fa_bwd_workspace_size": (_sz, [_p, _p, _i, _i, _i, _i, _i]),
    "fa_bwd": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p,
                    _i, _i, _i, _i, _i, _i, _f, _i, _p, _sz, _p]),
    "fa_bwd_gqa": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p,
                        _i, _i, _i, _i, _i, _i, _i, _f, _i, _p, _sz, _p]),
    "fa_bwd_ex": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p,
                       _i, _i, _i, _i, _i, _i, _i, _i, _f, _i, _p, _sz, _p]),
    "fa_bwd_lse": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p,
                        _i, _i, _i, _i, _i, _i, _i, _i, _f, _i, _p, _sz, _p]),
    "fa_bwd_dq_finalize": (_i, [_p, _p, _i, _i, _i, _f, _p]),
    "fa_bwd_noalloc": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p,
                            _i, _i, _i, _i, _i, _i, _f, _p]),
    "fa_selftest_wait_timeout": (_i, [_p]),
    "fa_check_device_status": (_i, [_p]),
    "fa_last_error": (ctypes.c_char_p, []),
}

_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Loads the library once and attaches the C signatures."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
            "(or python attention_backward_sm_gb300/build.py)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
