"""GPU parity of the joint key RMSNorm (reading note "Low-Rank Key Value
Attention", section 8) through the C ABI: the stored reciprocal norms
against the float64 oracle over the stored rows; decode (tensor-core and
generic kernels, bf16, fp32 and 8-bit caches) given those reciprocals; and
end to end (prefill on a history, the decode step, RoPE with norms, the
16 x 4096 workload) against the plain definition: RMS-normalised
materialised keys."""
import numpy as np
import pytest
import torch

import lrkv_inputs as I
import oracle
from oracle import norm as N
from oracle import rope as R
from gpu_util import DevDecode, assert_close, dev, host, host_bits, pools_f64

pytestmark = pytest.mark.gpu
EPS = 1e-6


def _norm_tol(adt):
    # one rounding of the stored reciprocal (bf16: 2^-9 relative) on top of
    # fp32 accumulation
    return 4e-3 if adt == "bf16" else 2e-6


def _all_rows(case):
    """(positions, seq_ids) of every visible row of the case."""
    pos = np.concatenate([np.arange(L) for L in case.seq_lens]).astype(np.int32)
    sid = np.concatenate([np.full(L, b) for b, L in enumerate(case.seq_lens)]).astype(np.int32)
    return pos, sid


def _with_norms(case):
    """DevDecode of the case with an N_K pool (canary-filled) written by
    lrkv_key_norms for every visible row."""
    import rank_kv_attention_gb300 as L
    adt = case.act_dtype
    dc = DevDecode(case)
    nk = np.full((case.num_pages, case.page_size, case.H),
                 I.BF16_NAN_BITS if adt == "bf16" else np.float32(np.nan),
                 dtype=np.uint16 if adt == "bf16" else np.float32)
    dc.cache.N_K = dev(nk, adt)
    dc.cache.norm_eps = EPS
    pos, sid = _all_rows(case)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.key_norms(dev(pos, "i32"), dev(sid, "i32"), dc.B_K, dc.cache, dc.page_table, status=st)
    assert int(st.item()) == 0
    return dc


def _stored_norms_f64(dc, adt):
    t = dc.cache.N_K
    return I.to_f64(host_bits(t), "bf16") if adt == "bf16" else host(t, "f32")


@pytest.mark.parametrize("H,d_h,r,dtype", [(16, 128, 48, "bf16"), (8, 64, 24, "bf16"),
                                           (4, 16, 4, "f32"), (16, 128, 48, "fp8")])
def test_key_norm_values(H, d_h, r, dtype):
    lens = [1, 17, 300, 65]
    case = I.make_decode_case(len(lens), H, d_h, r, lens, dtype=dtype, seed=H + r, shuffle=True,
                              spare_pages=2)
    dc = _with_norms(case)
    adt = case.act_dtype
    got = _stored_norms_f64(dc, adt)
    SK, SV, RK, RV = pools_f64(case)
    want = N.key_norms(SK.reshape(-1, d_h), RK.reshape(-1, H, r), I.to_f64(case.B_K, adt),
                       EPS).reshape(case.num_pages, case.page_size, H)
    vis = np.zeros((case.num_pages, case.page_size), bool)
    for b, L in enumerate(case.seq_lens):
        for t in range(L):
            vis[case.page_table[b, t // case.page_size], t % case.page_size] = True
    rel = np.abs(got[vis] - want[vis]) / want[vis]
    assert rel.max() <= _norm_tol(adt), rel.max()
    # slots that are not rows keep the canary
    assert np.all(np.isnan(got[~vis]))


LENS = [1, 17, 300, 64, 65, 129]


@pytest.mark.parametrize("H,d_h,r,dtype", [(16, 128, 48, "bf16"), (32, 128, 32, "bf16"),
                                           (16, 128, 56, "fp8"), (8, 64, 24, "bf16"),
                                           (4, 16, 4, "f32")])
def test_norm_decode_parity(H, d_h, r, dtype):
    """Decode given the stored reciprocals equals the oracle with the same
    reciprocals, and the plain definition (RMS-normalised keys) within the
    tolerance of one more rounding."""
    case = I.make_decode_case(len(LENS), H, d_h, r, LENS, dtype=dtype, seed=2 * H + r, shuffle=True,
                              spare_pages=2)
    dc = _with_norms(case)
    adt = case.act_dtype
    got = host(dc.run(), adt)
    f = lambda a: I.to_f64(a, adt)
    ref = N.decode_norm(f(case.q), *pools_f64(case), f(case.B_K), f(case.B_V),
                        _stored_norms_f64(dc, adt), case.page_table, case.seq_lens, case.page_size)
    assert_close(got, ref, adt, f"norm decode H={H} r={r} {dtype}")
    plain = np.stack([N.decode_request_norm(
        f(case.q[b]), *[oracle.gather_rows(p, case.page_table[b], L, case.page_size)
                        for p in pools_f64(case)], f(case.B_K), f(case.B_V), EPS)
        for b, L in enumerate(case.seq_lens)])
    assert_close(got, plain, adt, "against the plain definition")


def test_norm_decode_T4096_sampled():
    case = I.config_decode_case("decode_T4096")
    dc = _with_norms(case)
    got = host(dc.run(), "bf16")
    rng = np.random.default_rng(5)
    pairs = sorted({(b, int(rng.integers(case.H))) for b in range(case.B)})
    f = lambda a: I.to_f64(a, "bf16")
    ref = N.decode_norm(f(case.q), *pools_f64(case), f(case.B_K), f(case.B_V),
                        _stored_norms_f64(dc, "bf16"), case.page_table, case.seq_lens,
                        case.page_size, pairs=pairs)
    idx = tuple(np.array(pairs).T)
    assert_close(got[idx], ref[idx], "bf16", "decode_T4096 with norms")


def test_norm_prefill_and_decode_step():
    """Chunked prefill on a history, then a decode step, on a cache with
    norms: the library writes the norms of the rows it appends."""
    import rank_kv_attention_gb300 as L
    from rank_kv_attention_gb300.api import PagedCache
    H, d_h, r, d = 16, 128, 48, 256
    new, hist = [40, 90], [70, 5]
    caps = [a + b + 1 for a, b in zip(new, hist)]   # + the decode step's row
    rng = np.random.default_rng(7)
    pt, num_pages = I.make_page_table(caps, 64, True, rng, 2)
    pools = I.empty_pools(num_pages, 64, H, d_h, r, "bf16", canary=True)
    nk = np.full((num_pages, 64, H), I.BF16_NAN_BITS, np.uint16)
    cache = PagedCache(*[dev(p, "bf16") for p in pools], N_K=dev(nk, "bf16"), norm_eps=EPS)
    w = I.make_weights(d, H, d_h, r, "bf16", seed=8)
    draw = lambda n: I.f32_to_bf16_bits(rng.standard_normal((n, d)).astype(np.float32))
    Xh, Xn = draw(sum(hist)), draw(sum(new))
    Q = I.f32_to_bf16_bits(rng.standard_normal((sum(new), H, d_h)).astype(np.float32))
    pos_h = np.concatenate([np.arange(k) for k in hist]).astype(np.int32)
    sid_h = np.concatenate([np.full(k, b) for b, k in enumerate(hist)]).astype(np.int32)
    Wd = [dev(getattr(w, n), "bf16") for n in ("W_S_K", "W_S_V", "U_K", "U_V")]
    BK, BV = dev(w.B_K, "bf16"), dev(w.B_V, "bf16")
    ptd = dev(pt, "i32")
    L.append(dev(Xh, "bf16"), dev(pos_h, "i32"), dev(sid_h, "i32"), *Wd, cache, ptd)
    L.key_norms(dev(pos_h, "i32"), dev(sid_h, "i32"), BK, cache, ptd)
    assert L.prefill_kernel_kind(cache) == L.LRKV_PREFILL_PER_ROW
    cu = np.array([0, new[0], sum(new)], np.int32)
    out = L.prefill(dev(Xn, "bf16"), dev(Q, "bf16"), dev(cu, "i32"), dev(np.array(hist, np.int32), "i32"),
                    int(max(caps)), *Wd, BK, BV, cache, ptd)
    f = lambda a: I.to_f64(a, "bf16")
    stored = lambda: [f(host_bits(t)) for t in (cache.S_K, cache.S_V, cache.R_K, cache.R_V)]
    pos_n = np.concatenate([np.arange(hist[b], hist[b] + new[b]) for b in range(2)])
    sid_n = np.concatenate([np.full(new[b], b) for b in range(2)])
    ref = np.stack([N.decode_request_norm(
        f(Q[i]), *[oracle.gather_rows(p, pt[sid_n[i]], pos_n[i] + 1, 64) for p in stored()],
        f(w.B_K), f(w.B_V), EPS) for i in range(len(pos_n))])
    assert_close(host(out, "bf16"), ref, "bf16", "prefill with norms")
    # one decode step: the new rows' norms are written too
    lens = np.array([hist[b] + new[b] + 1 for b in range(2)], np.int32)
    Xs = draw(2)
    q = I.f32_to_bf16_bits(rng.standard_normal((2, H, d_h)).astype(np.float32))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out2 = L.decode_step(dev(Xs, "bf16"), *Wd, dev(q, "bf16"), cache, BK, BV, dev(lens, "i32"), ptd,
                         int(lens.max()), status=st)
    assert int(st.item()) == 0
    ref2 = np.stack([N.decode_request_norm(
        f(q[b]), *[oracle.gather_rows(p, pt[b], lens[b], 64) for p in stored()], f(w.B_K),
        f(w.B_V), EPS) for b in range(2)])
    assert_close(host(out2, "bf16"), ref2, "bf16", "decode step with norms")


def test_rope_with_norms():
    """The exact rotary embedding on a cache with norms: the rotation keeps a
    key's norm, so the score is (rotated score) x (stored reciprocal)."""
    import rank_kv_attention_gb300 as L
    lens = [5, 200, 64]
    case = I.make_decode_case(3, 16, 128, 48, lens, dtype="bf16", seed=12, shuffle=True)
    dc = _with_norms(case)
    table = L.rope_table(128, 200)
    got = host(L.decode_rope(dc.q, dc.cache, dc.B_K, dc.B_V, dc.seq_lens, dc.page_table, 200, table),
               "bf16")
    f = lambda a: I.to_f64(a, "bf16")
    ref = np.empty_like(got)
    for b, Lb in enumerate(lens):
        rows = [oracle.gather_rows(p, case.page_table[b], Lb, 64) for p in pools_f64(case)]
        for h in range(16):
            K = N.rms_normalise(oracle.expand_head(rows[0], rows[2][:, h], f(case.B_K[h])), EPS)
            V = oracle.expand_head(rows[1], rows[3][:, h], f(case.B_V[h]))
            ref[b, h] = oracle.attend(R.rotate(f(case.q[b, h]), Lb - 1),
                                      R.rotate(K, np.arange(Lb)), V)
    assert_close(got, ref, "bf16", "rope with norms")
