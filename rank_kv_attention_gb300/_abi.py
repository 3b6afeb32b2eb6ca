"""ctypes view of the C ABI in include/lrkv.h (argument marshalling only).

Loading fails loudly when ``liblrkv.so`` has not been built: there is no
fallback implementation of any kind.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "liblrkv.so")

LRKV_F32 = 0
LRKV_BF16 = 1
LRKV_FP8_E4M3 = 2

LRKV_OK = 0
LRKV_E_INVALID_ARG = -1
LRKV_E_SHAPE = -2
LRKV_E_DTYPE = -3
LRKV_E_BOUNDS = -4
LRKV_E_WORKSPACE = -5
LRKV_E_CUDA = -6

LRKV_NOALLOC_SCRATCH_BYTES = 16 << 20

LRKV_PREFILL_PER_ROW = 0
LRKV_PREFILL_TILED = 1

LRKV_PROFILE_ATTENTION = 0
LRKV_PROFILE_PROJECTION = 1
LRKV_PROFILE_SCORES = 2

LRKV_STATUS_BAD_PAGE = 1
LRKV_STATUS_BAD_SEQLEN = 2
LRKV_STATUS_BAD_ROW = 4
LRKV_STATUS_TIMEOUT = 8


class CacheDesc(ctypes.Structure):
    """Mirror of lrkv_cache_t."""
    _fields_ = [
        ("S_K", ctypes.c_void_p), ("S_V", ctypes.c_void_p),
        ("R_K", ctypes.c_void_p), ("R_V", ctypes.c_void_p),
        ("num_pages", ctypes.c_int32), ("page_size", ctypes.c_int32),
        ("H", ctypes.c_int32), ("d_h", ctypes.c_int32), ("r", ctypes.c_int32),
        ("dtype", ctypes.c_int32), ("scale", ctypes.c_float * 4),
        ("N_K", ctypes.c_void_p), ("norm_eps", ctypes.c_float),
        ("G", ctypes.c_int32),
    ]


class LrkvError(RuntimeError):
    def __init__(self, fn, code, lib=None):
        msg = f"{fn} failed: {code}"
        if lib is not None:
            msg += f" ({lib.lrkv_status_string(code).decode()})"
            if code == LRKV_E_CUDA:
                msg += f", cudaError {lib.lrkv_last_cuda_error()}"
        super().__init__(msg)
        self.code = code


_lib = None

P = ctypes.c_void_p
I32 = ctypes.c_int32
SZ = ctypes.c_size_t
CACHE_P = ctypes.POINTER(CacheDesc)

SIGNATURES = {
    "lrkv_append": (ctypes.c_int, [P, P, P, I32, I32, P, P, P, P, CACHE_P, P, I32, I32, P, P]),
    "lrkv_decode_workspace_bytes": (SZ, [I32, I32, I32, I32, I32, I32]),
    "lrkv_decode": (ctypes.c_int, [P, CACHE_P, P, P, P, P, I32, I32, I32, P, P, SZ, P, P]),
    "lrkv_decode_noalloc": (ctypes.c_int, [P, CACHE_P, P, P, P, P, I32, I32, I32, P, P, P]),
    "lrkv_decode_step_workspace_bytes": (SZ, [I32, I32, I32, I32, I32, I32]),
    "lrkv_decode_step": (ctypes.c_int, [P, I32, P, P, P, P, P, CACHE_P, P, P, P, P, I32, I32, I32, P,
                                        P, SZ, P, P]),
    "lrkv_decode_step_host_workspace_bytes": (SZ, [I32, I32, I32, I32, I32, I32, I32]),
    "lrkv_decode_step_host": (ctypes.c_int, [P, I32, P, P, P, P, P, CACHE_P, P, P, P, P, I32, I32, I32,
                                             P, P, SZ, P, P]),
    "lrkv_step_graph_create": (ctypes.c_int, [ctypes.POINTER(P), P, I32, P, P, P, P, P, CACHE_P, P, P,
                                              P, P, I32, I32, I32, P, P, SZ, P]),
    "lrkv_step_graph_launch": (ctypes.c_int, [P, P]),
    "lrkv_step_graph_destroy": (None, [P]),
    "lrkv_prefill_workspace_bytes": (SZ, [I32, I32, I32, I32, I32, I32, I32]),
    "lrkv_prefill": (ctypes.c_int, [P, P, P, P, I32, I32, I32, I32, P, P, P, P, P, P, CACHE_P, P,
                                    I32, P, P, SZ, P, P]),
    "lrkv_prefill_kernel_kind": (ctypes.c_int, [CACHE_P]),
    "lrkv_rope_table_bytes": (SZ, [I32, I32]),
    "lrkv_rope_table": (ctypes.c_int, [ctypes.c_double, I32, I32, P, P]),
    "lrkv_decode_rope_workspace_bytes": (SZ, [I32, I32, I32, I32, I32, I32]),
    "lrkv_key_norms": (ctypes.c_int, [P, P, I32, P, CACHE_P, P, I32, I32, P, P]),
    "lrkv_decode_rope": (ctypes.c_int, [P, CACHE_P, P, P, P, P, I32, I32, I32, P, I32, P, P, SZ, P,
                                        P]),
    "lrkv_prefill_rope": (ctypes.c_int, [P, P, P, P, I32, I32, I32, I32, P, P, P, P, P, P, CACHE_P,
                                         P, I32, P, I32, P, P, SZ, P, P]),
    "lrkv_cache_bytes": (SZ, [I32, I32, I32, ctypes.c_int64, I32]),
    "lrkv_cache_bytes_grouped": (SZ, [I32, I32, I32, I32, ctypes.c_int64, I32]),
    "lrkv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "lrkv_last_cuda_error": (ctypes.c_int, []),
    "lrkv_version": (ctypes.c_int, []),
    "lrkv_profile_enable": (ctypes.c_int, [ctypes.c_int]),
    "lrkv_profile_read": (ctypes.c_int, [I32, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(I32)]),
}


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def check(fn_name: str, code: int):
    if code != LRKV_OK:
        raise LrkvError(fn_name, code, lib())
