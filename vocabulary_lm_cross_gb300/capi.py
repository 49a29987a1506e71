"""ctypes declarations of libvlmce.so (the C ABI in include/vlmce.h).

Argument marshalling only.  The library must have been built (see
``vocabulary_lm_cross_gb300.build``); a missing library is an error, never a
fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

from .build import LIB

OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED_DTYPE = 2
ERR_MISALIGNED = 3
ERR_UNSUPPORTED_DEVICE = 4
ERR_WORKSPACE_TOO_SMALL = 5
ERR_CUDA = 6
ERR_TOO_LARGE = 7

F32 = 0
BF16 = 1
F16 = 2
NONE = 0
MEAN = 1
SUM = 2
DEVERR_TIMEOUT = 1

_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_f32 = ctypes.c_float
_sz = ctypes.c_size_t

# name -> (restype, argtypes); every function include/vlmce.h declares.
SIGNATURES = {
    "vlmce_status_string": (ctypes.c_char_p, [_i32]),
    "vlmce_last_error": (ctypes.c_char_p, []),
    "vlmce_ce_max_vocab": (_i64, [_i32]),
    "vlmce_profile_events": (None, [_vp, _vp]),
    "vlmce_ce_workspace_bytes": (_sz, [_i64, _i64, _i32]),
    "vlmce_ce_describe_plan": (_i32, [_i64, _i64, _i32, _f32, _i32, _vp]),
    "ce_fwd_bwd": (_i32, [_vp, _i32, _vp, _i64, _i64, _i64, _i64, _f32, _f32, _i32, _f32, _vp, _vp,
                          _vp, _vp, _vp, _sz, _vp]),
    "ce_fwd_bwd_ex": (_i32, [_vp, _i32, _vp, _i64, _i64, _i64, _i64, _f32, _f32, _i32, _f32, _vp,
                             _i32, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "ce_fwd_bwd_host": (_i32, [_vp, _i32, _vp, _i64, _i64, _i64, _i64, _f32, _f32, _i32, _f32, _vp,
                               _vp, _vp, _vp, _vp, _sz, _vp]),
    "vlmce_ce_host_workspace_bytes": (_sz, [_i64, _i64, _i64, _i32]),
    "ce_shard_stats": (_i32, [_vp, _i32, _vp, _i64, _i64, _i64, _i64, _i64, _f32, _vp, _vp]),
    "ce_merge_stats": (_i32, [_vp, _i32, _i64, _vp, _vp]),
    "ce_shard_fwd_bwd": (_i32, [_vp, _i32, _vp, _i64, _i64, _i64, _i64, _i64, _i64, _f32, _f32, _i32,
                                _f32, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "ce_shard_fwd_bwd_gathered": (_i32, [_vp, _i32, _vp, _i64, _i64, _i64, _i64, _i64, _i64, _f32,
                                         _f32, _i32, _f32, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _sz,
                                         _vp]),
    "swiglu_fwd": (_i32, [_vp, _i32, _i64, _i64, _i64, _vp, _i64, _vp]),
    "swiglu_bwd": (_i32, [_vp, _i64, _vp, _i64, _vp, _i64, _i32, _i64, _i64, _vp]),
    "ce_fwd_bwd_noalloc": (_i32, [_vp, _i32, _vp, _i64, _i64, _i64, _i64, _f32, _f32, _i32, _f32,
                                  _vp, _vp, _vp, _vp, _vp]),
    "vlmce_ce_noalloc_max_rows": (_i64, []),
    "vlmce_flce_workspace_bytes": (_sz, [_i64, _i64, _i64]),
    "flce_fwd_bwd": (_i32, [_vp, _i64, _vp, _i64, _vp, _i64, _i64, _i64, _i64, _f32, _f32, _i32,
                            _f32, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _sz, _vp]),
    "flce_fwd_bwd_ex": (_i32, [_vp, _i32, _i64, _vp, _i64, _vp, _i64, _i64, _i64, _i64, _f32, _f32,
                               _i32, _f32, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _vp, _sz, _vp]),
    "vlmce_flce_rows_workspace_bytes": (_sz, [_i64, _i64, _i64, _i64]),
    "flce_fwd_bwd_rows": (_i32, [_vp, _i32, _i64, _vp, _i64, _vp, _i64, _i64, _i64, _i64, _f32,
                                 _f32, _i32, _f32, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _vp,
                                 _sz, _vp]),
    "vlmce_gemm": (_i32, [_vp, _i32, _vp, _i32, _vp, _i64, _i64, _i64, _i64, _i64, _i64, _i32,
                          _i32, _vp]),
    "vlmce_gemm_bf16": (_i32, [_vp, _i32, _vp, _i32, _vp, _i64, _i64, _i64, _i64, _i64, _i64,
                               _i32, _vp]),
    "vlmce_flce_profile_events": (None, [_vp, _vp]),
}


class VlmceError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = ""
        if status == ERR_CUDA:
            detail = " [" + lib().vlmce_last_error().decode() + "]"
        super().__init__(f"{where}: {status_string(status)}{detail}")


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB):
                raise RuntimeError(
                    f"{LIB} is missing: build it with vocabulary_lm_cross_gb300.build.build() "
                    "(there is no CPU fallback)")
            handle = ctypes.CDLL(LIB)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib


def status_string(status: int) -> str:
    return lib().vlmce_status_string(int(status)).decode()


def check(status: int, where: str) -> None:
    if status != OK:
        raise VlmceError(status, where)
