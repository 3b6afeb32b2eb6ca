"""GPU parity of lrkv_prefill (through the C ABI): the tiny fp32 workload
(fresh 64-token prompt, then one appended row and a decode step), chunked
prefill on top of an existing history, and the 8 x 2048 prefill workload on
sampled rows and heads."""
import numpy as np
import pytest
import torch

import lrkv_inputs as I
import oracle
from gpu_util import assert_close, dev, host

pytestmark = pytest.mark.gpu


def _setup(cfg_B, n_per_seq, start_pos, d, H, d_h, r, dtype, seed, spare=2):
    from rank_kv_attention_gb300.api import PagedCache
    w = I.make_weights(d, H, d_h, r, dtype, seed=seed)
    caps = [s + n for s, n in zip(start_pos, n_per_seq)]
    rng = np.random.default_rng(seed + 1)
    pt, num_pages = I.make_page_table(caps, 64, True, rng, spare)
    pools = I.empty_pools(num_pages, 64, H, d_h, r, dtype, canary=True)
    return w, pt, num_pages, pools


def _run_prefill(X, Q, n_per_seq, start_pos, w, pt, pools, dtype, cache=None):
    import rank_kv_attention_gb300 as L
    from rank_kv_attention_gb300.api import PagedCache
    if cache is None:
        cache = PagedCache(*[dev(p, dtype) for p in pools])
    cu = np.concatenate([[0], np.cumsum(n_per_seq)]).astype(np.int32)
    max_ctx = int(max(s + n for s, n in zip(start_pos, n_per_seq)))
    out = L.prefill(dev(X, dtype), dev(Q, dtype), dev(cu, "i32"), dev(np.array(start_pos), "i32"),
                    max_ctx, dev(w.W_S_K, dtype), dev(w.W_S_V, dtype), dev(w.U_K, dtype),
                    dev(w.U_V, dtype), dev(w.B_K, dtype), dev(w.B_V, dtype), cache, dev(pt, "i32"))
    return out, cache


def test_tiny_fp32_prefill_then_decode():
    """1 layer, B=1, d=64, H=4, d_h=16, r=4: prefill 64 rows, then append the
    65th row and decode it (queries q = x W_Q, W_Q drawn after the others)."""
    import rank_kv_attention_gb300 as L
    c = I.CONFIGS["tiny_fp32"]
    d, H, d_h, r, T = c["d"], c["H"], c["d_h"], c["r"], c["T"]
    f = lambda a: I.to_f64(a, "f32")
    w, pt, num_pages, pools = _setup(1, [T + 1], [0], d, H, d_h, r, "f32", seed=c["seed"])
    rng = np.random.default_rng(c["seed"] + 17)
    X = (rng.standard_normal((T + 1, d)) / np.sqrt(d)).astype(np.float32)
    Q = np.einsum("nd,hcd->nhc", X.astype(np.float64), f(w.W_Q)).astype(np.float32)
    out, cache = _run_prefill(X[:T], Q[:T], [T], [0], w, pt, pools, "f32")
    pos = np.arange(T + 1)
    sid = np.zeros(T + 1, np.int64)
    ref = oracle.prefill(f(Q), f(X), pos, sid, f(w.W_S_K), f(w.W_S_V), f(w.U_K), f(w.U_V),
                         f(w.B_K), f(w.B_V))
    assert_close(host(out, "f32"), ref[:T], "f32", "prefill rows")
    # decode step: append row T, then attend over T + 1 rows
    L.append(dev(X[T:], "f32"), dev(np.array([T]), "i32"), dev(np.array([0]), "i32"),
             dev(w.W_S_K, "f32"), dev(w.W_S_V, "f32"), dev(w.U_K, "f32"), dev(w.U_V, "f32"),
             cache, dev(pt, "i32"))
    o = L.decode(dev(Q[T:], "f32"), cache, dev(w.B_K, "f32"), dev(w.B_V, "f32"),
                 dev(np.array([T + 1]), "i32"), dev(pt, "i32"), T + 1)
    assert_close(host(o, "f32")[0], ref[T], "f32", "decode step")


@pytest.mark.parametrize("dtype,H,d_h,r", [("bf16", 16, 128, 48), ("f32", 4, 32, 8)])
def test_chunked_prefill_on_history(dtype, H, d_h, r):
    """Two requests with earlier history (appended first) and a new chunk."""
    d = 96
    hist, new = [70, 5], [33, 90]
    w, pt, num_pages, pools = _setup(2, new, hist, d, H, d_h, r, dtype, seed=21)
    rng = np.random.default_rng(5)
    draw = lambda s: (rng.standard_normal(s) * (1 / np.sqrt(d))).astype(np.float32)
    enc = (lambda a: I.f32_to_bf16_bits(a)) if dtype == "bf16" else (lambda a: a)
    Xh = [enc(draw((k, d))) for k in hist]
    Xn = enc(draw((sum(new), d)))
    Qn = enc(rng.standard_normal((sum(new), H, d_h)).astype(np.float32))
    import rank_kv_attention_gb300 as L
    from rank_kv_attention_gb300.api import PagedCache
    cache = PagedCache(*[dev(p, dtype) for p in pools])
    # history through lrkv_prefill too (its outputs unused here)
    for b in range(2):
        cu = np.array([0] * (b + 1) + [hist[b]] * (2 - b), np.int32)
        Qh = np.zeros((hist[b], H, d_h), np.uint16 if dtype == "bf16" else np.float32)
        _run_prefill(Xh[b], Qh, [hist[b] if i == b else 0 for i in range(2)], [0, 0], w, pt, pools,
                     dtype, cache=cache)
    out, _ = _run_prefill(Xn, Qn, new, hist, w, pt, pools, dtype, cache=cache)
    f = lambda a: I.to_f64(a, dtype)
    history = {}
    for b in range(2):
        history[b] = oracle.project(f(Xh[b]), f(w.W_S_K), f(w.W_S_V), f(w.U_K), f(w.U_V))
    pos = np.concatenate([np.arange(hist[b], hist[b] + new[b]) for b in range(2)])
    sid = np.concatenate([np.full(new[b], b) for b in range(2)])
    ref = oracle.prefill(f(Qn), f(Xn), pos, sid, f(w.W_S_K), f(w.W_S_V), f(w.U_K), f(w.U_V),
                         f(w.B_K), f(w.B_V), history=history)
    assert_close(host(out, dtype), ref, dtype, "chunked prefill")


def test_prefill_2048_sampled():
    """8 fresh 2048-token prompts, d=2048, H=16, d_h=128, r=48; oracle on
    sampled rows of two requests (all earlier rows of those requests are
    projected by the oracle)."""
    c = I.CONFIGS["prefill_2048"]
    Bq, d, H, d_h, r, T = c["B"], c["d"], c["H"], c["d_h"], c["r"], c["T"]
    ac = I.make_append_case([T] * Bq, [0] * Bq, d, dtype="bf16", seed=c["seed"], shuffle=True)
    w = I.make_weights(d, H, d_h, r, "bf16", seed=c["seed"])
    rng = np.random.default_rng(99)
    Q = I.f32_to_bf16_bits(rng.standard_normal((Bq * T, H, d_h)).astype(np.float32))
    pools = I.empty_pools(ac.num_pages, 64, H, d_h, r, "bf16", canary=True)
    out, _ = _run_prefill(ac.X, Q, [T] * Bq, [0] * Bq, w, ac.page_table, pools, "bf16")
    got = host(out, "bf16")
    f = lambda a: I.to_f64(a, "bf16")
    for b in (0, 5):
        rows = np.arange(b * T, (b + 1) * T)
        want_rows = sorted({0, 1, 63, 64, 1000, T - 1} | set(rng.integers(0, T, 6).tolist()))
        heads = sorted(set(rng.integers(0, H, 3).tolist()) | {0, H - 1})
        ref = oracle.prefill(f(Q[rows]), f(ac.X[rows]), ac.positions[rows], ac.seq_ids[rows],
                             f(w.W_S_K), f(w.W_S_V), f(w.U_K), f(w.U_V), f(w.B_K), f(w.B_V),
                             rows_wanted=want_rows, heads_wanted=heads)
        for i in want_rows:
            assert_close(got[rows[i]][heads], ref[i][heads], "bf16", f"req {b} row {i}")


# --------------------------------------------------------------------------
# Tiled tensor-core attention: shapes, tails, history, bad pages
# --------------------------------------------------------------------------
def _history_then_prefill(H, r, page_size, hist, new, seed, d=64, d_h=128, bad_page=None):
    """Append each request's history with lrkv_append, then lrkv_prefill the
    new rows.  Returns (device out, status, float64 oracle out, per-row
    request ids, per-row positions, cache)."""
    import rank_kv_attention_gb300 as L
    from rank_kv_attention_gb300.api import PagedCache
    w = I.make_weights(d, H, d_h, r, "bf16", seed=seed)
    rng = np.random.default_rng(seed + 1)
    caps = [a + b for a, b in zip(hist, new)]
    pt, num_pages = I.make_page_table(caps, page_size, True, rng, 2)
    pools = I.empty_pools(num_pages, page_size, H, d_h, r, "bf16", canary=True)
    cache = PagedCache(*[dev(p, "bf16") for p in pools])
    assert L.prefill_kernel_kind(cache) == L.LRKV_PREFILL_TILED
    draw = lambda s: I.f32_to_bf16_bits((rng.standard_normal(s) / np.sqrt(d)).astype(np.float32))
    Xh = [draw((k, d)) for k in hist]
    if sum(hist):
        pos = np.concatenate([np.arange(k) for k in hist]).astype(np.int32)
        sid = np.concatenate([np.full(k, b) for b, k in enumerate(hist)]).astype(np.int32)
        L.append(dev(np.concatenate(Xh), "bf16"), dev(pos, "i32"), dev(sid, "i32"),
                 dev(w.W_S_K, "bf16"), dev(w.W_S_V, "bf16"), dev(w.U_K, "bf16"),
                 dev(w.U_V, "bf16"), cache, dev(pt, "i32"))
    if bad_page is not None:
        b, k = bad_page
        pt = pt.copy()
        pt[b, k] = num_pages + 7
    Xn = draw((sum(new), d))
    Qn = I.f32_to_bf16_bits(rng.standard_normal((sum(new), H, d_h)).astype(np.float32))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    cu = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    max_ctx = int(max(caps))
    out = L.prefill(dev(Xn, "bf16"), dev(Qn, "bf16"), dev(cu, "i32"), dev(np.array(hist), "i32"),
                    max_ctx, dev(w.W_S_K, "bf16"), dev(w.W_S_V, "bf16"), dev(w.U_K, "bf16"),
                    dev(w.U_V, "bf16"), dev(w.B_K, "bf16"), dev(w.B_V, "bf16"), cache,
                    dev(pt, "i32"), status=status)
    f = lambda a: I.to_f64(a, "bf16")
    history = {b: oracle.project(f(Xh[b]), f(w.W_S_K), f(w.W_S_V), f(w.U_K), f(w.U_V))
               for b in range(len(hist)) if hist[b]}
    pos = np.concatenate([np.arange(hist[b], hist[b] + new[b]) for b in range(len(new))])
    sid = np.concatenate([np.full(new[b], b) for b in range(len(new))])
    ref = oracle.prefill(f(Qn), f(Xn), pos, sid, f(w.W_S_K), f(w.W_S_V), f(w.U_K), f(w.U_V),
                         f(w.B_K), f(w.B_V), history=history)
    return out, int(status.item()), ref, sid, pos, cache


# (H, r, page_size, history, new rows): several query tiles per request,
# ragged last tiles and key tiles, an empty request, r not a multiple of 16,
# r = 8 and 64, H r below one 64-column box, 128-row pages.
TILED = [
    (16, 48, 64, [0, 77, 200], [300, 1, 129]),
    (8, 8, 64, [5, 0], [140, 64]),
    (4, 16, 128, [130, 0, 64], [70, 200, 0]),
    (32, 32, 64, [64, 1], [64, 255]),
    (16, 56, 64, [10, 300], [90, 40]),
    (2, 64, 128, [0], [257]),
    (16, 40, 64, [33], [200]),
    (1, 48, 64, [0], [100]),
]


@pytest.mark.parametrize("H,r,page_size,hist,new", TILED)
def test_tiled_prefill_parity(H, r, page_size, hist, new):
    out, st, ref, _, _, _ = _history_then_prefill(H, r, page_size, hist, new, seed=H * 7 + r)
    assert st == 0
    assert_close(host(out, "bf16"), ref, "bf16", f"H={H} r={r} page={page_size}")


def test_tiled_prefill_deterministic():
    a, _, _, _, _, _ = _history_then_prefill(16, 48, 64, [40], [300], seed=3)
    b, _, _, _, _, _ = _history_then_prefill(16, 48, 64, [40], [300], seed=3)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_tiled_prefill_bad_page_flagged():
    """Request 1's second page id is outside the pool: append and attention
    skip it and flag LRKV_STATUS_BAD_PAGE; request 0 and request 1's rows
    that see only its first page still match the oracle; all outputs stay
    finite."""
    import rank_kv_attention_gb300 as L
    out, st, ref, sid, pos, _ = _history_then_prefill(16, 48, 64, [0, 0], [100, 150], seed=12,
                                                      bad_page=(1, 1))
    got = host(out, "bf16")
    assert st & L.LRKV_STATUS_BAD_PAGE
    assert np.all(np.isfinite(got))
    keep = (sid == 0) | (pos < 64)
    assert_close(got[keep], ref[keep], "bf16", "rows unaffected by the bad page")


def test_prefill_2048_pools_full():
    """The four pools lrkv_prefill writes for the whole 8 x 2048 workload
    (16384 rows, d = 2048, 128 x 7 output tiles of the persistent projection)
    against the float64 projection placed by the oracle: every written slot
    within the bf16 tolerance and, tighter, equal to the oracle's value
    rounded to bf16 except where the tensor core's fp32 accumulation (not a
    correctly rounded sum: ~1e-6 relative over d = 2048 products) lands on
    the other side of a rounding boundary -- at most 0.5% of the slots, each
    within one bf16 unit of |ref| (2^-7 relative) plus 1e-6 absolute
    (projections are ~0.02 in magnitude; the floor covers values that cancel
    to near zero, where fp32 and float64 may even round to opposite signs);
    spare pages keep their NaN canary."""
    c = I.CONFIGS["prefill_2048"]
    Bq, d, H, d_h, r, T = c["B"], c["d"], c["H"], c["d_h"], c["r"], c["T"]
    ac = I.make_append_case([T] * Bq, [0] * Bq, d, dtype="bf16", seed=c["seed"], shuffle=True,
                            spare_pages=2)
    w = I.make_weights(d, H, d_h, r, "bf16", seed=c["seed"])
    rng = np.random.default_rng(99)
    Q = I.f32_to_bf16_bits(rng.standard_normal((Bq * T, H, d_h)).astype(np.float32))
    pools = I.empty_pools(ac.num_pages, 64, H, d_h, r, "bf16", canary=True)
    _, cache = _run_prefill(ac.X, Q, [T] * Bq, [0] * Bq, w, ac.page_table, pools, "bf16")
    f = lambda a: I.to_f64(a, "bf16")
    rows = oracle.project(f(ac.X), f(w.W_S_K), f(w.W_S_V), f(w.U_K), f(w.U_V))
    want = oracle.place([f(p) for p in pools], rows, ac.positions, ac.seq_ids, ac.page_table, 64)
    touched = np.zeros((ac.num_pages, 64), bool)
    for b, p in zip(ac.seq_ids, ac.positions):
        touched[ac.page_table[b, p // 64], p % 64] = True
    assert touched.sum() == Bq * T and (~touched).sum() == 2 * 64
    from gpu_util import host_bits
    for k, t in enumerate((cache.S_K, cache.S_V, cache.R_K, cache.R_V)):
        got_bits = host_bits(t)
        got = I.bf16_bits_to_f64(got_bits)
        assert_close(got[touched], want[k][touched], "bf16", f"pool {k}")
        ref = want[k][touched]
        off = got_bits[touched] != I.f32_to_bf16_bits(ref.astype(np.float32))
        assert np.count_nonzero(off) <= 5e-3 * off.size, f"pool {k}: {np.count_nonzero(off)} off"
        e = np.abs(got[touched][off] - ref[off])
        assert np.all(e <= 2.0 ** -7 * np.abs(ref[off]) + 1e-6), f"pool {k}: worst {e.max():.3e}"
        assert np.all(got_bits[~touched] == I.BF16_NAN_BITS), f"pool {k} canary"
