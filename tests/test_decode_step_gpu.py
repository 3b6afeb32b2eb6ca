"""GPU parity of lrkv_decode_step (through the C ABI): each request's new row
lands where lrkv_append would put it (position seq_lens[b] - 1), nothing else
in the cache changes, and the output matches the float64 oracle's
append-then-decode.  Covers the tensor-core decode shapes, shapes that run
the generic kernels, a request whose only row is the new one, more than 64
requests (the many-row append kernel), invalid lengths and pages, and the
16 x 4096 decode workload.  The append kernels take each row's place from the
lengths and the decode's prologue runs beside the append."""
import numpy as np
import pytest
import torch

import lrkv_inputs as I
import oracle
from gpu_util import DevDecode, assert_close, dev, host, host_bits

pytestmark = pytest.mark.gpu


def _step_case(H, d_h, r, lens, d, dtype, seed, page_size=64, spare=2):
    """A decode case whose new-row slots (position L-1) hold canaries, new rows
    X ~ N(0, 1) (so their projections are as large as the cached rows) and
    projection weights N(0, 1/d)."""
    case = I.make_decode_case(len(lens), H, d_h, r, lens, dtype=dtype, seed=seed, shuffle=True,
                              spare_pages=spare, page_size=page_size)
    w = I.make_weights(d, H, d_h, r, dtype, seed=seed + 1)
    rng = np.random.default_rng(seed + 2)
    Xf = rng.standard_normal((len(lens), d)).astype(np.float32)
    X = I.f32_to_bf16_bits(Xf) if dtype == "bf16" else Xf
    canary = I.BF16_NAN_BITS if dtype == "bf16" else I.F32_NAN_CANARY
    for pool in (case.S_K, case.S_V, case.R_K, case.R_V):
        for b, L in enumerate(case.seq_lens):
            if L >= 1:
                pool[case.page_table[b, (L - 1) // page_size], (L - 1) % page_size] = canary
    return case, w, X


def _oracle(case, w, X, valid=None):
    """float64 append of the new rows (stored at the cache's precision), then
    the float64 decode over every request's seq_lens rows."""
    f = lambda a: I.to_f64(a, case.dtype)
    S_K, S_V, R_K, R_V = oracle.project(f(X), f(w.W_S_K), f(w.W_S_V), f(w.U_K), f(w.U_V))
    rows = [S_K, S_V, R_K, R_V]
    if case.dtype == "bf16":  # the cache stores each value once, rounded to bf16
        rows = [I.bf16_bits_to_f64(I.f32_to_bf16_bits(x.astype(np.float32))) for x in rows]
    keep = np.flatnonzero(case.seq_lens >= 1 if valid is None else valid)
    pools = oracle.place([f(p) for p in (case.S_K, case.S_V, case.R_K, case.R_V)],
                         [x[keep] for x in rows], case.seq_lens[keep] - 1, keep, case.page_table,
                         case.page_size)
    return pools


def _run_step(case, w, X, d_case=None):
    import rank_kv_attention_gb300 as L
    dc = d_case or DevDecode(case)
    dt = case.dtype
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = L.decode_step(dev(X, dt), dev(w.W_S_K, dt), dev(w.W_S_V, dt), dev(w.U_K, dt),
                        dev(w.U_V, dt), dc.q, dc.cache, dc.B_K, dc.B_V, dc.seq_lens, dc.page_table,
                        dc.max_seq_len, status=st)
    return out, dc, int(st.item())


def _check_cache(case, dc, pools, new_slots):
    """New-row slots hold the oracle's projections; every other slot keeps its
    original bytes."""
    for k, (orig, t) in enumerate(zip((case.S_K, case.S_V, case.R_K, case.R_V),
                                      (dc.cache.S_K, dc.cache.S_V, dc.cache.R_K, dc.cache.R_V))):
        got = host(t, case.dtype)
        assert_close(got[new_slots], pools[k][new_slots], case.dtype, f"pool {k} new rows")
        bits = host_bits(t)
        want = np.asarray(orig).view(bits.dtype)
        assert np.array_equal(bits[~new_slots], want[~new_slots]), f"pool {k} other slots"


def _new_slots(case, which=None):
    m = np.zeros((case.num_pages, case.page_size), bool)
    for b, L in enumerate(case.seq_lens):
        if L >= 1 and (which is None or which[b]):
            m[case.page_table[b, (L - 1) // case.page_size], (L - 1) % case.page_size] = True
    return m


LENS = [1, 17, 300, 64, 65, 129]


# (H, r, d): shapes the tensor-core decode covers
@pytest.mark.parametrize("H,r,d", [(16, 48, 2048), (32, 32, 256), (16, 64, 256), (16, 16, 512),
                                   (16, 56, 384)])
def test_decode_step_tensor_core_parity(H, r, d):
    case, w, X = _step_case(H, 128, r, LENS, d, "bf16", seed=H * 100 + r + d)
    out, dc, st = _run_step(case, w, X)
    assert st == 0
    pools = _oracle(case, w, X)
    _check_cache(case, dc, pools, _new_slots(case))
    f = lambda a: I.to_f64(a, "bf16")
    ref = oracle.decode(f(case.q), *pools, f(case.B_K), f(case.B_V), case.page_table,
                        case.seq_lens, case.page_size)
    assert_close(host(out, "bf16"), ref, "bf16", f"H={H} r={r} d={d}")


# d not a multiple of 32 (the FMA few-row append), d_h != 128 (the generic
# decode), an fp32 cache and 32-row pages
@pytest.mark.parametrize("H,d_h,r,d,dtype,ps", [(16, 128, 48, 136, "bf16", 64),
                                                (8, 64, 24, 256, "bf16", 64),
                                                (4, 16, 4, 64, "f32", 64),
                                                (16, 128, 48, 256, "bf16", 32)])
def test_decode_step_other_shapes(H, d_h, r, d, dtype, ps):
    case, w, X = _step_case(H, d_h, r, LENS, d, dtype, seed=7 + H + r, page_size=ps)
    out, dc, st = _run_step(case, w, X)
    assert st == 0
    pools = _oracle(case, w, X)
    _check_cache(case, dc, pools, _new_slots(case))
    f = lambda a: I.to_f64(a, dtype)
    ref = oracle.decode(f(case.q), *pools, f(case.B_K), f(case.B_V), case.page_table,
                        case.seq_lens, case.page_size)
    assert_close(host(out, dtype), ref, dtype, f"H={H} d_h={d_h} r={r} d={d} {dtype} ps={ps}")


def test_decode_step_many_requests():
    """70 requests: the step's rows go through the many-row (tcgen05) append
    kernel with places taken from the lengths."""
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(1, 200, size=70)]
    case, w, X = _step_case(16, 128, 48, lens, 256, "bf16", seed=53)
    out, dc, st = _run_step(case, w, X)
    assert st == 0
    pools = _oracle(case, w, X)
    _check_cache(case, dc, pools, _new_slots(case))
    f = lambda a: I.to_f64(a, "bf16")
    ref = oracle.decode(f(case.q), *pools, f(case.B_K), f(case.B_V), case.page_table,
                        case.seq_lens, case.page_size)
    assert_close(host(out, "bf16"), ref, "bf16", "70 requests")


def test_decode_step_equals_append_then_decode():
    """The step and lrkv_append + lrkv_decode agree (same inputs, two copies
    of the cache)."""
    import rank_kv_attention_gb300 as L
    lens = [5, 900, 64, 1, 333]
    case, w, X = _step_case(16, 128, 48, lens, 1024, "bf16", seed=31)
    out_f, dc_f, _ = _run_step(case, w, X)
    dc = DevDecode(case)
    pos = dev((case.seq_lens - 1).astype(np.int32), "i32")
    ids = dev(np.arange(len(lens), dtype=np.int32), "i32")
    L.append(dev(X, "bf16"), pos, ids, dev(w.W_S_K, "bf16"), dev(w.W_S_V, "bf16"),
             dev(w.U_K, "bf16"), dev(w.U_V, "bf16"), dc.cache, dc.page_table)
    out_s = dc.run()
    assert_close(host(out_f, "bf16"), host(out_s, "bf16"), "bf16", "step vs separate")
    for a, b in zip((dc_f.cache.S_K, dc_f.cache.R_V), (dc.cache.S_K, dc.cache.R_V)):
        assert_close(host(a, "bf16")[_new_slots(case)], host(b, "bf16")[_new_slots(case)], "bf16")


@pytest.mark.parametrize("H,r,d", [(16, 48, 2048), (16, 48, 136)])
def test_decode_step_bad_length_and_page(H, r, d):
    """Request 0 has length 0 (no new row, out = 0, BAD_SEQLEN).  Request 2's
    new row is the first row of a page whose id is out of range: it is not
    written, not attended (BAD_PAGE), and request 2 equals the decode of its
    older rows.  Request 1 is untouched."""
    import rank_kv_attention_gb300 as L
    lens = [0, 70, 129]
    case, w, X = _step_case(H, 128, r, lens, d, "bf16", seed=41, spare=1)
    case.page_table = case.page_table.copy()
    bad = case.page_table[2, 2]
    case.page_table[2, 2] = case.num_pages + 3  # position 128 = row 0 of page 2
    out, dc, st = _run_step(case, w, X)
    assert st & L.LRKV_STATUS_BAD_SEQLEN and st & L.LRKV_STATUS_BAD_PAGE
    got = host(out, "bf16")
    assert np.all(got[0] == 0) and np.all(np.isfinite(got))
    ok = np.array([False, True, False])
    pools = _oracle(case, w, X, valid=ok)
    f = lambda a: I.to_f64(a, "bf16")
    lens_seen = np.array([0, 70, 128], np.int32)  # request 2 without its new row
    ref = oracle.decode(f(case.q), *pools, f(case.B_K), f(case.B_V), case.page_table, lens_seen,
                        case.page_size, pairs=[(b, h) for b in (1, 2) for h in range(H)])
    assert_close(got[1:], ref[1:], "bf16", "valid requests")
    # the invalid page was never written: its real slot still holds the canary
    assert np.all(host_bits(dc.cache.S_K)[bad, 0] == I.BF16_NAN_BITS)


def test_decode_step_T4096_sampled():
    """The 16 x 4096 decode workload through lrkv_decode_step (d = 2048), on
    sampled (request, head) outputs and every new row."""
    case = I.config_decode_case("decode_T4096")
    w = I.make_weights(2048, case.H, case.d_h, case.r, "bf16", seed=77)
    rng = np.random.default_rng(78)
    X = I.f32_to_bf16_bits(rng.standard_normal((case.B, 2048)).astype(np.float32))
    for pool in (case.S_K, case.S_V, case.R_K, case.R_V):
        for b, L in enumerate(case.seq_lens):
            pool[case.page_table[b, (L - 1) // case.page_size], (L - 1) % case.page_size] = \
                I.BF16_NAN_BITS
    out, dc, st = _run_step(case, w, X)
    assert st == 0
    pools = _oracle(case, w, X)
    _check_cache(case, dc, pools, _new_slots(case))
    pairs = sorted({(b, int(rng.integers(case.H))) for b in range(case.B)} | {(0, 0), (15, 15)})
    f = lambda a: I.to_f64(a, "bf16")
    ref = oracle.decode(f(case.q), *pools, f(case.B_K), f(case.B_V), case.page_table,
                        case.seq_lens, case.page_size, pairs=pairs)
    idx = tuple(np.array(pairs).T)
    assert_close(host(out, "bf16")[idx], ref[idx], "bf16", "decode_T4096 step")


@pytest.mark.parametrize("dtype,H,d_h,r,d,pinned", [("bf16", 16, 128, 48, 2048, True),
                                                    ("f32", 4, 16, 4, 64, True),
                                                    ("bf16", 16, 128, 48, 2048, False)])
def test_decode_step_host_buffers(dtype, H, d_h, r, d, pinned):
    """lrkv_decode_step_host (X, q, lengths and out in host memory) gives the
    same bits as lrkv_decode_step on device copies of the same inputs, in the
    output and in the cache, and matches the oracle.  Page-locked buffers go
    through their device-mapped addresses (a copy kernel in, the combine's
    stores out), pageable ones through the copy engines."""
    import rank_kv_attention_gb300 as L
    lens = [5, 900, 64, 1, 333]
    case, w, X = _step_case(H, d_h, r, lens, d, dtype, seed=61)
    out_d, dc_d, st_d = _run_step(case, w, X)
    dc = DevDecode(case)
    pin = (lambda t: t.pin_memory()) if pinned else (lambda t: t.clone())
    hX = pin(host_tensor(X, dtype))
    hq = pin(dc.q.cpu())
    hl = pin(torch.from_numpy(np.ascontiguousarray(case.seq_lens, dtype=np.int32)))
    ho = pin(torch.full(tuple(dc.q.shape), float("nan"), dtype=dc.q.dtype))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out_h = L.decode_step_host(hX, dev(w.W_S_K, dtype), dev(w.W_S_V, dtype), dev(w.U_K, dtype),
                               dev(w.U_V, dtype), hq, dc.cache, dc.B_K, dc.B_V, hl, dc.page_table,
                               dc.max_seq_len, out=ho, status=st)
    torch.cuda.synchronize()
    assert out_h is ho and out_h.is_pinned() == pinned
    assert int(st.item()) == 0 and st_d == 0
    assert torch.equal(out_h.view(torch.int16 if dtype == "bf16" else torch.int32),
                       out_d.cpu().view(torch.int16 if dtype == "bf16" else torch.int32))
    for a, b in zip((dc.cache.S_K, dc.cache.S_V, dc.cache.R_K, dc.cache.R_V),
                    (dc_d.cache.S_K, dc_d.cache.S_V, dc_d.cache.R_K, dc_d.cache.R_V)):
        assert np.array_equal(host_bits(a), host_bits(b))
    pools = _oracle(case, w, X)
    f = lambda a: I.to_f64(a, dtype)
    ref = oracle.decode(f(case.q), *pools, f(case.B_K), f(case.B_V), case.page_table,
                        case.seq_lens, case.page_size)
    assert_close(host(out_h, dtype), ref, dtype, f"host step {dtype}")


def host_tensor(a, kind):
    """A pinned host tensor of an array of bf16 bits or fp32 values."""
    if kind == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).pin_memory()


def test_step_graph_replays_with_new_inputs():
    """A step graph recorded once and launched for two consecutive steps,
    with the pinned inputs refilled in between (new rows, new queries,
    lengths + 1), gives the same bits as lrkv_decode_step_host called for the
    same two steps on a second copy of the cache, and matches the oracle."""
    import rank_kv_attention_gb300 as L
    lens = [5, 900, 64, 1, 333]
    H, d_h, r, d = 16, 128, 48, 2048
    case, w, X = _step_case(H, d_h, r, [x + 1 for x in lens], d, "bf16", seed=71)
    rng = np.random.default_rng(72)
    X2 = I.f32_to_bf16_bits(rng.standard_normal(X.shape).astype(np.float32))
    q2 = I.f32_to_bf16_bits(rng.standard_normal(case.q.shape).astype(np.float32))
    steps = [(X, case.q, np.array(lens, np.int32)), (X2, q2, np.array(lens, np.int32) + 1)]
    Wd = [dev(getattr(w, n), "bf16") for n in ("W_S_K", "W_S_V", "U_K", "U_V")]
    dg, dh = DevDecode(case), DevDecode(case)
    hX, hq = host_tensor(X, "bf16"), host_tensor(case.q, "bf16")
    hl = torch.zeros(len(lens), dtype=torch.int32).pin_memory()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = L.StepGraph(hX, *Wd, hq, dg.cache, dg.B_K, dg.B_V, hl, dg.page_table, dg.max_seq_len,
                    status=st)
    outs = []
    for Xs, qs, ls in steps:
        hX.copy_(host_tensor(Xs, "bf16"))
        hq.copy_(host_tensor(qs, "bf16"))
        hl.copy_(torch.from_numpy(ls))
        g.launch()
        torch.cuda.synchronize()
        ref = L.decode_step_host(host_tensor(Xs, "bf16"), *Wd, host_tensor(qs, "bf16"), dh.cache,
                                 dh.B_K, dh.B_V, torch.from_numpy(ls).pin_memory(), dh.page_table,
                                 dh.max_seq_len, status=st)
        torch.cuda.synchronize()
        assert torch.equal(g.out.view(torch.int16), ref.view(torch.int16))
        outs.append(host(g.out, "bf16"))
    g.close()
    assert int(st.item()) == 0
    for a, b in zip((dg.cache.S_K, dg.cache.R_V), (dh.cache.S_K, dh.cache.R_V)):
        assert np.array_equal(host_bits(a), host_bits(b))
    # the oracle: both steps' rows appended, then the second step's decode
    f = lambda a: I.to_f64(a, "bf16")
    pools = [f(p) for p in (case.S_K, case.S_V, case.R_K, case.R_V)]
    for Xs, _, ls in steps:
        rows = oracle.project(f(Xs), f(w.W_S_K), f(w.W_S_V), f(w.U_K), f(w.U_V))
        rows = [I.bf16_bits_to_f64(I.f32_to_bf16_bits(x.astype(np.float32))) for x in rows]
        pools = oracle.place(pools, rows, ls - 1, np.arange(len(lens)), case.page_table,
                             case.page_size)
    ref = oracle.decode(f(q2), *pools, f(case.B_K), f(case.B_V), case.page_table, steps[1][2],
                        case.page_size)
    assert_close(outs[1], ref, "bf16", "graph step 2")
