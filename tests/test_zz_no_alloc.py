"""lrkv_decode_noalloc: the decode entry point for callers that cannot
allocate device memory (a host that reserves all HBM for its own pool, or a
plugin hook that forbids allocation).  It must give the same result as
lrkv_decode with a caller-provided workspace, call after call, while its
scratch lives in the library's own device array.

Called through the C ABI (ctypes), like a C caller would.  This file is
collected last so that a stop-at-first-failure run has already run every
other test before it.
"""
import ctypes

import numpy as np
import pytest
import torch

import lrkv_inputs as I
from gpu_util import DevDecode, assert_close, host, oracle_decode

pytestmark = pytest.mark.gpu


def _noalloc(lib, d, out, status=None):
    desc = d.cache.desc()
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    return lib.lrkv_decode_noalloc(
        P(d.q), ctypes.byref(desc), P(d.B_K), P(d.B_V), P(d.seq_lens), P(d.page_table),
        d.case.B, d.page_table.shape[1], d.max_seq_len, P(out),
        None if status is None else P(status), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("H,d_h,r,lens", [
    (16, 128, 48, [1, 300, 2000, 65, 4096]),   # tensor-core split kernel
    (4, 64, 24, [7, 129, 900]),                # generic split kernel
])
def test_noalloc_matches_workspace_decode_twice(H, d_h, r, lens):
    import rank_kv_attention_gb300 as L
    lib = L.lib()
    case = I.make_decode_case(len(lens), H, d_h, r, lens, seed=31 + r, shuffle=True, spare_pages=2)
    d = DevDecode(case)
    ref = d.run()                                  # lrkv_decode with its own workspace
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):                          # two calls in a row share the scratch array
        out = torch.full_like(ref, float("nan"))
        assert _noalloc(lib, d, out, status) == L.LRKV_OK
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert_close(host(out, "bf16"), host(ref, "bf16"), "bf16", f"call {call}")
    assert_close(host(out, "bf16"), oracle_decode(case), "bf16", "vs oracle")


def test_noalloc_rejects_sizes_beyond_its_array():
    import rank_kv_attention_gb300 as L
    lib = L.lib()
    # enough requests that the scratch would exceed LRKV_NOALLOC_SCRATCH_BYTES
    B, H, d_h, r = 6000, 32, 128, 64
    need = lib.lrkv_decode_workspace_bytes(B, H, d_h, r, 64, L.LRKV_BF16)
    assert need > L._abi.LRKV_NOALLOC_SCRATCH_BYTES
    desc = L.CacheDesc(256, 256, 256, 256, 8, 64, H, d_h, r, L.LRKV_BF16)
    rc = lib.lrkv_decode_noalloc(256, ctypes.byref(desc), 256, 256, 256, 256, B, 1, 64, 256,
                                 None, None)
    assert rc == L.LRKV_E_WORKSPACE
