"""Host-side checks of the C-ABI library: it builds, loads, exports every
function include/lrkv.h declares, and its host-only entry points (sizes,
status strings, argument validation that rejects before any CUDA work)
behave as documented.  No call here touches a GPU."""
import ctypes
from fractions import Fraction
import os
import re

import pytest

import oracle
from oracle import grouped
from rank_kv_attention_gb300 import _abi
from rank_kv_attention_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return _abi.lib()


def header_functions():
    txt = open(os.path.join(ROOT, "include", "lrkv.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"LRKV_API\s+[\w\s\*]*?\b(lrkv_\w+)\s*\(", txt)))


def test_exports_every_declared_symbol(lib):
    names = header_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_abi.SIGNATURES), "binding and header disagree"


def test_version_and_strings(lib):
    assert lib.lrkv_version() >= 100
    assert lib.lrkv_status_string(0) == b"ok"
    assert b"workspace" in lib.lrkv_status_string(_abi.LRKV_E_WORKSPACE)


@pytest.mark.parametrize("H,d_h,r,T,dt,eb", [(16, 128, 48, 4096, 1, 2), (32, 128, 32, 32768, 1, 2),
                                             (4, 16, 4, 65, 0, 4), (18, 128, 56, 2048, 1, 2),
                                             (16, 128, 48, 4096, 2, 1), (32, 64, 8, 100, 2, 1)])
def test_cache_bytes_is_equation_9(lib, H, d_h, r, T, dt, eb):
    got = lib.lrkv_cache_bytes(H, d_h, r, T, dt)
    assert got == oracle.lrkv_payload(eb, 1, 1, T, H, d_h, r)


def test_cache_bytes_rejects_bad_shapes(lib):
    assert lib.lrkv_cache_bytes(0, 128, 48, 10, 1) == 0
    assert lib.lrkv_cache_bytes(16, 130, 48, 10, 1) == 0   # bf16 needs d_h % 8 == 0
    assert lib.lrkv_cache_bytes(16, 128, 48, 10, 7) == 0   # bad dtype
    assert lib.lrkv_cache_bytes(16, 120, 48, 10, 2) == 0   # 8-bit codes need d_h % 16 == 0
    assert lib.lrkv_cache_bytes(3, 128, 8, 10, 2) == 0     # ... and H * r % 16 == 0


@pytest.mark.parametrize("H,d_h,r,G,T,dt,eb", [(16, 128, 32, 2, 4096, 1, 2), (32, 128, 32, 8, 100, 1, 2),
                                               (4, 16, 4, 4, 65, 0, 4), (16, 128, 48, 1, 7, 2, 1)])
def test_cache_bytes_grouped(lib, H, d_h, r, G, T, dt, eb):
    """Equation 9 with G shared rows per token: 2 T (G d_h + H r) elements;
    the oracle's grouped payload ratio times the multi-head bytes."""
    got = lib.lrkv_cache_bytes_grouped(H, d_h, r, G, T, dt)
    assert got == 2 * T * (G * d_h + H * r) * eb
    assert Fraction(got, 2 * T * H * d_h * eb) == grouped.payload_ratio_grouped(H, d_h, r, G)
    if G == 1:
        assert got == lib.lrkv_cache_bytes(H, d_h, r, T, dt)


def test_cache_groups_checked_on_host(lib):
    assert lib.lrkv_cache_bytes_grouped(16, 128, 48, 3, 10, 1) == 0    # G must divide H
    assert lib.lrkv_cache_bytes_grouped(16, 128, 48, 0, 10, 1) == 0
    assert lib.lrkv_cache_bytes_grouped(16, 128, 48, 32, 10, 1) == 0   # G <= H
    ws = ctypes.c_void_p(256)

    def call(cache):
        return lib.lrkv_decode(16, ctypes.byref(cache), 16, 16, 16, 16, 2, 4, 100, 16, ws, 1 << 30, None,
                               None)
    assert call(_cache(G=3)) == _abi.LRKV_E_SHAPE
    assert call(_cache(G=-1)) == _abi.LRKV_E_SHAPE
    assert call(_cache(G=32)) == _abi.LRKV_E_SHAPE


def test_fp8_cache_scales_checked_on_host(lib):
    """An 8-bit cache needs four positive, finite scales with finite reciprocals."""
    ws = ctypes.c_void_p(256)

    def call(scale):
        c = _cache(dtype=_abi.LRKV_FP8_E4M3)
        c.scale = (ctypes.c_float * 4)(*scale)
        return lib.lrkv_decode(16, ctypes.byref(c), 16, 16, 16, 16, 2, 4, 100, 16, ws, 1 << 30,
                               None, None)
    for bad in ((0.0, 1, 1, 1), (1, -1, 1, 1), (1, 1, float("inf"), 1), (1, 1, 1, float("nan")),
                (1, 1, 1, 1e-45)):
        assert call(bad) == _abi.LRKV_E_DTYPE, bad


def test_workspace_sizes_positive_and_monotone(lib):
    a = lib.lrkv_decode_workspace_bytes(16, 16, 128, 48, 4096, 1)
    b = lib.lrkv_decode_workspace_bytes(64, 16, 128, 48, 4096, 1)
    assert 0 < a < b
    assert lib.lrkv_decode_workspace_bytes(0, 16, 128, 48, 4096, 1) == 0
    assert lib.lrkv_prefill_workspace_bytes(8, 16384, 16, 128, 48, 2048, 1) > 0


def _cache(dtype=1, **kw):
    c = _abi.CacheDesc(16, 16, 16, 16, 4, 64, 16, 128, 48, dtype)  # fake aligned addresses
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def test_decode_rejects_on_host(lib):
    ws = ctypes.c_void_p(256)
    good = dict(q=16, BK=16, BV=16, sl=16, pt=16, B=2, mp=4, msl=100, out=16, ws=ws, wsb=1 << 30)

    def call(cache, **over):
        a = dict(good, **over)
        return lib.lrkv_decode(a["q"], ctypes.byref(cache), a["BK"], a["BV"], a["sl"], a["pt"], a["B"],
                               a["mp"], a["msl"], a["out"], a["ws"], a["wsb"], None, None)
    assert call(_cache(), q=None) == _abi.LRKV_E_INVALID_ARG
    assert call(_cache(), q=8) == _abi.LRKV_E_INVALID_ARG           # misaligned
    assert call(_cache(dtype=5)) == _abi.LRKV_E_DTYPE
    assert call(_cache(d_h=130)) == _abi.LRKV_E_SHAPE
    assert call(_cache(page_size=40)) == _abi.LRKV_E_SHAPE
    assert call(_cache(), msl=4 * 64 + 1) == _abi.LRKV_E_BOUNDS     # beyond max_pages * page_size
    assert call(_cache(), B=0) == _abi.LRKV_E_SHAPE
    assert call(_cache(), ws=None) == _abi.LRKV_E_WORKSPACE
    assert call(_cache(), ws=ctypes.c_void_p(16)) == _abi.LRKV_E_WORKSPACE   # not 256-aligned
    assert call(_cache(), wsb=16) == _abi.LRKV_E_WORKSPACE
    assert lib.lrkv_decode(16, None, 16, 16, 16, 16, 2, 4, 100, 16, ws, 1 << 30, None, None) \
        == _abi.LRKV_E_INVALID_ARG


def test_append_rejects_on_host(lib):
    c = _cache()
    ok_args = [16, 16, 16, 5, 2048, 16, 16, 16, 16, ctypes.byref(c), 16, 2, 4, None, None]
    a = list(ok_args); a[0] = None
    assert lib.lrkv_append(*a) == _abi.LRKV_E_INVALID_ARG
    a = list(ok_args); a[4] = 2047          # d not a multiple of 8 for bf16
    assert lib.lrkv_append(*a) == _abi.LRKV_E_SHAPE
    a = list(ok_args); a[3] = -1
    assert lib.lrkv_append(*a) == _abi.LRKV_E_SHAPE
    a = list(ok_args); a[3] = 0             # n == 0 is a no-op, even with null rows
    a[0] = None
    assert lib.lrkv_append(*a) == _abi.LRKV_OK


def test_prefill_rejects_on_host(lib):
    c = _cache()
    args = [16, 16, 16, 16, 2, 10, 300, 2048, 16, 16, 16, 16, 16, 16, ctypes.byref(c), 16, 4, 16,
            ctypes.c_void_p(256), 1 << 30, None, None]
    assert lib.lrkv_prefill(*args) == _abi.LRKV_E_BOUNDS   # max_ctx 300 > 4 pages * 64
    args[6] = 200
    args[18] = None
    assert lib.lrkv_prefill(*args) == _abi.LRKV_E_WORKSPACE


def test_prefill_kernel_kind_host_checks(lib):
    assert lib.lrkv_prefill_kernel_kind(None) == _abi.LRKV_E_INVALID_ARG
    assert lib.lrkv_prefill_kernel_kind(ctypes.byref(_cache(dtype=5))) == _abi.LRKV_E_DTYPE
    assert lib.lrkv_prefill_kernel_kind(ctypes.byref(_cache(d_h=130))) == _abi.LRKV_E_SHAPE
    # shapes outside the tiled kernel always take the per-row path
    assert lib.lrkv_prefill_kernel_kind(ctypes.byref(_cache(d_h=64))) == _abi.LRKV_PREFILL_PER_ROW
    assert lib.lrkv_prefill_kernel_kind(ctypes.byref(_cache(r=72))) == _abi.LRKV_PREFILL_PER_ROW
    assert lib.lrkv_prefill_kernel_kind(ctypes.byref(_cache(page_size=32))) == \
        _abi.LRKV_PREFILL_PER_ROW
    assert lib.lrkv_prefill_kernel_kind(ctypes.byref(_cache(dtype=0))) == _abi.LRKV_PREFILL_PER_ROW
    # covered shape: tiled wherever the driver can encode tensor maps
    assert lib.lrkv_prefill_kernel_kind(ctypes.byref(_cache())) in (
        _abi.LRKV_PREFILL_PER_ROW, _abi.LRKV_PREFILL_TILED)


def test_decode_step_rejects_on_host(lib):
    ws = ctypes.c_void_p(256)

    def call(**over):
        a = dict(X=16, d=2048, W=16, q=16, c=_cache(), BK=16, BV=16, sl=16, pt=16, B=2, mp=4,
                 msl=100, out=16, ws=ws, wsb=1 << 30)
        a.update(over)
        return lib.lrkv_decode_step(a["X"], a["d"], a["W"], a["W"], a["W"], a["W"], a["q"],
                                    ctypes.byref(a["c"]), a["BK"], a["BV"], a["sl"], a["pt"],
                                    a["B"], a["mp"], a["msl"], a["out"], a["ws"], a["wsb"], None,
                                    None)
    assert call(X=None) == _abi.LRKV_E_INVALID_ARG
    assert call(W=None) == _abi.LRKV_E_INVALID_ARG
    assert call(q=None) == _abi.LRKV_E_INVALID_ARG
    assert call(d=2047) == _abi.LRKV_E_SHAPE             # bf16 rows need d % 8 == 0
    assert call(c=_cache(dtype=3)) == _abi.LRKV_E_DTYPE
    assert call(msl=4 * 64 + 1) == _abi.LRKV_E_BOUNDS     # beyond max_pages * page_size
    assert call(ws=None) == _abi.LRKV_E_WORKSPACE
    assert call(wsb=64) == _abi.LRKV_E_WORKSPACE
    a = lib.lrkv_decode_step_workspace_bytes(16, 16, 128, 48, 4096, 1)
    assert a >= lib.lrkv_decode_workspace_bytes(16, 16, 128, 48, 4096, 1) > 0
    assert lib.lrkv_decode_step_workspace_bytes(0, 16, 128, 48, 4096, 1) == 0


def test_decode_step_host_rejects_on_host(lib):
    """The host-buffer step checks everything before it enqueues a copy; its
    host buffers need no alignment, its workspace holds the step's plus the
    device copies of X, q, the lengths and out."""
    ws = ctypes.c_void_p(256)

    def call(**over):
        a = dict(X=3, d=2048, W=16, q=5, c=_cache(), BK=16, BV=16, sl=7, pt=16, B=2, mp=4,
                 msl=100, out=9, ws=ws, wsb=1 << 30)
        a.update(over)
        return lib.lrkv_decode_step_host(a["X"], a["d"], a["W"], a["W"], a["W"], a["W"], a["q"],
                                         ctypes.byref(a["c"]), a["BK"], a["BV"], a["sl"], a["pt"],
                                         a["B"], a["mp"], a["msl"], a["out"], a["ws"], a["wsb"],
                                         None, None)
    for k in ("X", "q", "sl", "out", "W", "BK", "pt"):
        assert call(**{k: None}) == _abi.LRKV_E_INVALID_ARG, k
    assert call(BK=8) == _abi.LRKV_E_INVALID_ARG           # device bases stay 16-byte aligned
    assert call(d=2047) == _abi.LRKV_E_SHAPE
    assert call(msl=4 * 64 + 1) == _abi.LRKV_E_BOUNDS
    assert call(ws=None) == _abi.LRKV_E_WORKSPACE
    assert call(ws=ctypes.c_void_p(272)) == _abi.LRKV_E_WORKSPACE   # 256-byte alignment
    need = lib.lrkv_decode_step_host_workspace_bytes(2, 16, 128, 48, 2048, 100, 1)
    assert call(wsb=need - 1) == _abi.LRKV_E_WORKSPACE
    step = lib.lrkv_decode_step_workspace_bytes(2, 16, 128, 48, 100, 1)
    # + X (2 x 2048), q and out (2 x 16 x 128) bf16, lengths: each rounded to 256 bytes
    assert need == step + 8192 + 8192 + 256 + 8192
    assert lib.lrkv_decode_step_host_workspace_bytes(2, 16, 128, 48, 0, 100, 1) == 0


def test_step_graph_checks_before_recording(lib):
    """lrkv_step_graph_create checks its arguments like the host step before
    it touches a stream (so these run without a GPU); NULL handles are
    refused or ignored."""
    ws = ctypes.c_void_p(256)
    h = ctypes.c_void_p(12345)

    def create(**over):
        a = dict(X=3, d=2048, W=16, q=5, c=_cache(), BK=16, BV=16, sl=7, pt=16, B=2, mp=4,
                 msl=100, out=9, ws=ws, wsb=1 << 30)
        a.update(over)
        return lib.lrkv_step_graph_create(ctypes.byref(h), a["X"], a["d"], a["W"], a["W"], a["W"],
                                          a["W"], a["q"], ctypes.byref(a["c"]), a["BK"], a["BV"],
                                          a["sl"], a["pt"], a["B"], a["mp"], a["msl"], a["out"],
                                          a["ws"], a["wsb"], None)
    assert create(X=None) == _abi.LRKV_E_INVALID_ARG and h.value is None
    h.value = 12345
    assert create(sl=None) == _abi.LRKV_E_INVALID_ARG and h.value is None
    assert create(msl=4 * 64 + 1) == _abi.LRKV_E_BOUNDS
    assert create(wsb=1024) == _abi.LRKV_E_WORKSPACE
    assert lib.lrkv_step_graph_create(None, 3, 2048, 16, 16, 16, 16, 5, ctypes.byref(_cache()), 16,
                                      16, 7, 16, 2, 4, 100, 9, ws, 1 << 30, None) == \
        _abi.LRKV_E_INVALID_ARG
    assert lib.lrkv_step_graph_launch(None, None) == _abi.LRKV_E_INVALID_ARG
    lib.lrkv_step_graph_destroy(None)


def test_rope_host_checks(lib):
    """Rotary entry points reject bad tables and shapes before any launch."""
    E = _abi
    assert lib.lrkv_rope_table(1.0, 128, 10, 256, None) == E.LRKV_E_INVALID_ARG     # base <= 1
    assert lib.lrkv_rope_table(float("inf"), 128, 10, 256, None) == E.LRKV_E_INVALID_ARG
    assert lib.lrkv_rope_table(1e4, 127, 10, 256, None) == E.LRKV_E_SHAPE           # odd d_h
    assert lib.lrkv_rope_table(1e4, 128, 0, 256, None) == E.LRKV_E_SHAPE
    assert lib.lrkv_rope_table(1e4, 128, 10, None, None) == E.LRKV_E_INVALID_ARG
    assert lib.lrkv_rope_table(1e4, 128, 10, 4, None) == E.LRKV_E_INVALID_ARG       # misaligned
    assert lib.lrkv_rope_table(1e4, 128, 10, 8, None) == E.LRKV_E_INVALID_ARG       # not 16-aligned
    # float pairs, then f16 pairs from the next 256-byte boundary
    assert lib.lrkv_rope_table_bytes(128, 10) == 5120 + 2560
    assert lib.lrkv_rope_table_bytes(2, 3) == 256 + 12
    assert lib.lrkv_rope_table_bytes(127, 10) == 0 and lib.lrkv_rope_table_bytes(128, 0) == 0
    # the rotary decode workspace holds the decode one plus operands and scores
    rb = lib.lrkv_decode_rope_workspace_bytes(16, 16, 128, 48, 4096, 1)
    assert rb >= lib.lrkv_decode_workspace_bytes(16, 16, 128, 48, 4096, 1) + 16 * 4096 * 16 * 4
    assert lib.lrkv_decode_rope_workspace_bytes(0, 16, 128, 48, 4096, 1) == 0
    ws = ctypes.c_void_p(256)

    def dec(cache, table=16, max_pos=100, msl=100):
        return lib.lrkv_decode_rope(16, ctypes.byref(cache), 16, 16, 16, 16, 2, 4, msl, table,
                                    max_pos, 16, ws, 1 << 30, None, None)
    assert dec(_cache(), table=None) == E.LRKV_E_INVALID_ARG
    assert dec(_cache(), table=24) == E.LRKV_E_INVALID_ARG                        # not 16-aligned
    assert dec(_cache(), max_pos=99) == E.LRKV_E_BOUNDS                           # table too short
    assert dec(_cache(r=72)) == E.LRKV_E_SHAPE                                    # r > 64
    assert dec(_cache(d_h=130)) == E.LRKV_E_SHAPE
    assert dec(_cache(dtype=5)) == E.LRKV_E_DTYPE
    assert lib.lrkv_prefill_rope(16, 16, 16, 16, 2, 10, 100, 256, 16, 16, 16, 16, 16, 16,
                                 ctypes.byref(_cache()), 16, 4, 16, 99, 16, ws, 1 << 30, None,
                                 None) == E.LRKV_E_BOUNDS


def test_key_norm_host_checks(lib):
    """The joint key norm pool and eps are validated with the cache."""
    E = _abi
    ws = ctypes.c_void_p(256)

    def dec(cache):
        return lib.lrkv_decode(16, ctypes.byref(cache), 16, 16, 16, 16, 2, 4, 100, 16, ws, 1 << 30,
                               None, None)
    assert dec(_cache(N_K=8)) == E.LRKV_E_INVALID_ARG                     # misaligned
    assert dec(_cache(N_K=16, norm_eps=-1.0)) == E.LRKV_E_INVALID_ARG
    assert dec(_cache(N_K=16, norm_eps=float("nan"))) == E.LRKV_E_INVALID_ARG
    # lrkv_key_norms needs the pool
    assert lib.lrkv_key_norms(16, 16, 4, 16, ctypes.byref(_cache()), 16, 2, 4, None, None) \
        == E.LRKV_E_INVALID_ARG
    assert lib.lrkv_key_norms(16, 16, -1, 16, ctypes.byref(_cache(N_K=16)), 16, 2, 4, None, None) \
        == E.LRKV_E_SHAPE
    assert lib.lrkv_key_norms(16, 16, 0, 16, ctypes.byref(_cache(N_K=16)), 16, 2, 4, None, None) \
        == E.LRKV_OK
    assert lib.lrkv_key_norms(16, 16, 4, 8, ctypes.byref(_cache(N_K=16)), 16, 2, 4, None, None) \
        == E.LRKV_E_INVALID_ARG                                             # B_K misaligned
