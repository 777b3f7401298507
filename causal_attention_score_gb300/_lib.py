"""Loads libcsa_gb300.so and declares its C ABI (include/csa.h) for ctypes.

The library is built in-tree by ``build_lib.build()``. There is no fallback:
if the library is missing or fails to load, every operation raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build_lib

CSA_OK = 0
CSA_ERR_NULL = -1
CSA_ERR_SHAPE = -2
CSA_ERR_ALIGN = -3
CSA_ERR_UNSUPPORTED = -4
CSA_ERR_ARCH = -5
CSA_ERR_LAUNCH = -6
CSA_ERR_TIMEOUT = -7
CSA_ERR_CUDA = -8
CSA_ERR_CHECK = -9
CSA_ERR_WORKSPACE = -10
CSA_ERR_BUSY = -11

CSA_MASK_NAN = 0x7FC00000
CSA_MASK_NEG_INF = 0xFF800000
CSA_TRIMUL_FULL = 0
CSA_TRIMUL_LOWER_ONLY = 1

# name -> (restype, argtypes); mirrors include/csa.h
_vp = ctypes.c_void_p
_i = ctypes.c_int
_u32 = ctypes.c_uint32
SIGNATURES = {
    "trimul_forward": (_i, [_vp, _vp, _i, _i, _i, _i]),
    "trimul_forward_ex": (_i, [_vp, _vp, _i, _i, _i, _i, _u32, _u32, _vp]),
    "trimul_forward_noalloc": (_i, [_vp, _vp, _i, _i, _i, _i, _u32, _u32, _vp]),
    "trimul_forward_f32": (_i, [_vp, _vp, _i, _i, _i, _i, _u32, _u32, _vp]),
    "dense_xwt": (_i, [_vp, _vp, _vp, _i, _i, _i]),
    "batch_matmul_nt": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _vp]),
    "causal_softmax_forward": (_i, [_vp, _vp, _i, _i, _i, _i, _vp]),
    "dense_xwt_ex": (_i, [_vp, _vp, _vp, _i, _i, _i, _vp]),
    "dense_xwt_workspace_size": (_i, [_vp, _vp, _i, _i, _i, ctypes.POINTER(ctypes.c_size_t)]),
    "dense_xwt_ws": (_i, [_vp, _vp, _vp, _i, _i, _i, _vp, ctypes.c_size_t, _vp]),
    "dense_xwt_grouped": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _vp]),
    "dense_xwt_grouped_workspace_size": (_i, [_vp, _vp, _vp, _i, _i, _i,
                                              ctypes.POINTER(ctypes.c_size_t)]),
    "dense_xwt_grouped_ws": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _vp, ctypes.c_size_t, _vp]),
    "csa_get_status": (_i, [_vp]),
    "csa_status_string": (ctypes.c_char_p, [_i]),
    "csa_last_error": (ctypes.c_char_p, []),
    "csa_version": (ctypes.c_char_p, []),
    "csa_set_wait_limit_ns": (None, [ctypes.c_uint64]),
    "csa_get_wait_limit_ns": (ctypes.c_uint64, []),
    "csa_debug_inject": (None, [_i]),
    "csa_debug_hold_stream": (_i, [_vp]),
    "csa_debug_release_streams": (None, []),
    "csa_set_dense_fetch": (_i, [_i]),
    "csa_dense_tiling": (_i, [_i, _i, _i, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]),
    "csa_set_stream_sm_limit": (_i, [_vp, _i]),
    "csa_get_stream_sm_limit": (_i, [_vp, ctypes.POINTER(ctypes.c_int)]),
}


class CsaError(RuntimeError):
    def __init__(self, code: int, where: str, detail: str):
        self.code = code
        super().__init__(f"{where}: status {code} ({detail})")


_lib = None
_lock = threading.Lock()


def lib_path() -> str:
    return build_lib.LIBPATH


def load(path: str | None = None):
    """The loaded library (ctypes.CDLL). Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or lib_path()
            if not os.path.exists(p):
                raise RuntimeError(
                    f"CUDA extension {p} is not built; run causal_attention_score_gb300.build_lib.build()")
            if path is None and not build_lib.up_to_date(p):
                raise RuntimeError(
                    f"CUDA extension {p} was not built from the sources beside it (its "
                    f"{os.path.basename(build_lib.stamp_path(p))} does not match); run "
                    "causal_attention_score_gb300.build_lib.build()")
            lib = ctypes.CDLL(p)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
        return _lib


def check(code: int, where: str) -> None:
    if code != CSA_OK:
        lib = load()
        detail = lib.csa_last_error().decode() or lib.csa_status_string(code).decode()
        raise CsaError(code, where, detail)
