"""GB300-native (sm_103a) Low-Rank Key Value attention: factored-cache decode,
cache append and prefill as a C-ABI CUDA library (``liblrkv.so``) with a thin
PyTorch binding.

The C ABI is declared in ``include/lrkv.h``; ``api`` marshals torch tensors
into it.  Importing this package does not load the library; the first call
does, and raises if the library has not been built (see ``build.build``).
"""
from ._abi import (LRKV_BF16, LRKV_F32, LRKV_OK, LRKV_E_INVALID_ARG, LRKV_E_SHAPE,
                   LRKV_E_DTYPE, LRKV_E_BOUNDS, LRKV_E_WORKSPACE, LRKV_E_CUDA,
                   LRKV_STATUS_BAD_PAGE, LRKV_STATUS_BAD_SEQLEN, LRKV_STATUS_BAD_ROW,
                   LRKV_STATUS_TIMEOUT, LRKV_PREFILL_PER_ROW, LRKV_PREFILL_TILED, CacheDesc,
                   LrkvError, lib)

__all__ = [
    "lib", "CacheDesc", "LrkvError", "PagedCache", "append", "decode", "prefill",
    "decode_workspace_bytes", "prefill_workspace_bytes", "cache_bytes", "workspace",
    "prefill_kernel_kind", "decode_step", "decode_step_workspace_bytes", "rope_table",
    "decode_rope", "prefill_rope", "key_norms", "RopeTable", "rope_table_bytes",
    "decode_rope_workspace_bytes", "decode_step_host", "decode_step_host_workspace_bytes",
    "StepGraph",
]


def __getattr__(name):
    # torch-facing helpers are imported lazily so that the ctypes layer works
    # without importing torch
    if name in ("PagedCache", "append", "decode", "prefill", "decode_workspace_bytes",
                "prefill_workspace_bytes", "cache_bytes", "workspace", "prefill_kernel_kind",
                "decode_step", "decode_step_workspace_bytes", "rope_table", "decode_rope",
                "prefill_rope", "key_norms", "RopeTable", "rope_table_bytes",
                "decode_rope_workspace_bytes", "decode_step_host",
                "decode_step_host_workspace_bytes", "StepGraph"):
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
