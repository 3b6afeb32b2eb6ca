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
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import lrkv_inputs as I
from gpu_util import DevDecode, assert_close, host, oracle_decode

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


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
    """A batch whose scratch would not fit the built-in array is refused
    before anything is enqueued.  Every pointer passed is a real device
    buffer of the stated shape (valid lengths, valid page ids), so the call
    would be a correct decode even if the size check were ever skipped."""
    import rank_kv_attention_gb300 as L
    from rank_kv_attention_gb300.api import PagedCache
    lib = L.lib()
    B, H, d_h, r, page = 6000, 32, 128, 64, 64
    need = lib.lrkv_decode_workspace_bytes(B, H, d_h, r, page, L.LRKV_BF16)
    assert need > L._abi.LRKV_NOALLOC_SCRATCH_BYTES
    cache = PagedCache.empty(8, page, H, d_h, r, torch.bfloat16, "cuda")
    for t in (cache.S_K, cache.S_V, cache.R_K, cache.R_V):
        t.zero_()
    q = torch.zeros((B, H, d_h), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(q)
    BK = torch.zeros((H, d_h, r), dtype=torch.bfloat16, device="cuda")
    BV = torch.zeros_like(BK)
    seq_lens = torch.ones(B, dtype=torch.int32, device="cuda")
    pt = torch.zeros((B, 1), dtype=torch.int32, device="cuda")
    desc = cache.desc()
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = lib.lrkv_decode_noalloc(P(q), ctypes.byref(desc), P(BK), P(BV), P(seq_lens), P(pt), B, 1,
                                 page, P(out), None,
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert rc == L.LRKV_E_WORKSPACE


# The first call of a fresh process on its device loads the library's device
# code, which commits the built-in array and gives it an address; the child
# below makes lrkv_decode_noalloc that first library call and checks its
# output against lrkv_decode's, then calls it once more.
_CHILD = r"""
import ctypes, sys
import numpy as np
import torch
sys.path[:0] = [sys.argv[1], sys.argv[1] + "/tests"]
import lrkv_inputs as I
from gpu_util import DevDecode, assert_close, host
import rank_kv_attention_gb300 as L
lib = L.lib()
torch.cuda.set_device(0)
case = I.make_decode_case(3, 16, 128, 48, [5, 777, 1500], seed=77, shuffle=True, spare_pages=1)
d = DevDecode(case)
P = lambda t: ctypes.c_void_p(t.data_ptr())
s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
outs = []
for call in range(2):
    out = torch.full_like(d.q, float("nan"))
    desc = d.cache.desc()
    rc = lib.lrkv_decode_noalloc(P(d.q), ctypes.byref(desc), P(d.B_K), P(d.B_V), P(d.seq_lens),
                                 P(d.page_table), case.B, d.page_table.shape[1], d.max_seq_len,
                                 P(out), None, s)
    assert rc == 0, rc
    torch.cuda.synchronize()
    outs.append(out)
ref = d.run()
torch.cuda.synchronize()
for k, o in enumerate(outs):
    assert_close(host(o, "bf16"), host(ref, "bf16"), "bf16", f"fresh-process call {k}")
print("noalloc first call ok")
"""


def test_noalloc_first_call_in_a_fresh_process():
    r = subprocess.run([sys.executable, "-c", _CHILD, ROOT], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "noalloc first call ok" in r.stdout
