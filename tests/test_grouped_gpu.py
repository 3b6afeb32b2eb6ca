"""GPU parity of the grouped shared basis (reading note "Low-Rank Key Value
Attention", section 3 after equations 2-5: one shared basis per group of
heads) through the C ABI, against the float64 oracle: decode on the
tensor-core kernel (two groups) and the generic one (other group counts,
fp32 and 8-bit caches), append with exact placement and values, the per-row
prefill and the decode step, the rotary embedding and joint key norms with
groups, and the 16 x 4096 two-group workload sampled."""
import numpy as np
import pytest
import torch

import lrkv_inputs as I
import oracle
from oracle import grouped
from oracle import norm as N
from oracle import rope as R
from gpu_util import DevDecode, assert_close, dev, host, host_bits, oracle_decode, pools_f64

pytestmark = pytest.mark.gpu

LENS = [1, 2, 17, 300, 64, 65, 129, 900]


@pytest.mark.parametrize("H,d_h,r,G,dtype,ps", [(16, 128, 48, 2, "bf16", 64), (16, 128, 32, 2, "bf16", 32),
                                                (16, 128, 48, 4, "bf16", 64), (8, 64, 24, 2, "bf16", 16),
                                                (4, 16, 4, 2, "f32", 64), (16, 128, 48, 2, "fp8", 64),
                                                (32, 128, 32, 8, "bf16", 32), (4, 32, 8, 4, "f32", 16)])
def test_grouped_decode_parity(H, d_h, r, G, dtype, ps):
    case = I.make_decode_case(len(LENS), H, d_h, r, LENS, dtype=dtype, seed=H + r + G, shuffle=True,
                              spare_pages=2, page_size=ps, groups=G)
    got = host(DevDecode(case).run(), case.act_dtype)
    assert_close(got, oracle_decode(case), case.act_dtype, f"H={H} r={r} G={G} {dtype}")


def test_grouped_decode_T4096_sampled():
    """The 16 x 4096 workload with two groups (the bench's decode_T4096_g2)."""
    case = I.config_decode_case("decode_T4096_g2")
    got = host(DevDecode(case).run(), "bf16")
    rng = np.random.default_rng(10)
    pairs = sorted({(b, int(rng.integers(case.H))) for b in range(case.B)} | {(0, 7), (0, 8), (15, 15)})
    ref = oracle_decode(case, pairs)
    idx = tuple(np.array(pairs).T)
    assert_close(got[idx], ref[idx], "bf16", "decode_T4096_g2")


@pytest.mark.parametrize("n_per_seq", [[37, 1, 130, 64], [3, 1, 2]])
def test_grouped_append_exact(n_per_seq):
    """Integer-valued rows and {-1, 0, 1} weights with two groups: the written
    bytes equal the oracle's placement of its projections bit for bit (the
    many-row and the few-row kernels), untouched slots keep the canary."""
    import rank_kv_attention_gb300 as L
    from rank_kv_attention_gb300.api import PagedCache
    H, d_h, r, d, G = 16, 128, 48, 256, 2
    ac = I.make_append_case(n_per_seq, [0, 500, 63, 64][:len(n_per_seq)], d, dtype="bf16", seed=1,
                            shuffle=True, spare_pages=2, interleave=True)
    rng = np.random.default_rng(2)
    ac.X = I.f32_to_bf16_bits(rng.integers(-3, 4, size=ac.X.shape).astype(np.float32))
    w = I.make_weights(d, H, d_h, r, "bf16", seed=3, groups=G)
    for name in ("W_S_K", "W_S_V", "U_K", "U_V"):
        a = getattr(w, name)
        vals = rng.integers(-1, 2, size=a.shape).astype(np.float32) * (rng.random(a.shape) < 0.1)
        setattr(w, name, I.f32_to_bf16_bits(vals))
    pools = I.empty_pools(ac.num_pages, ac.page_size, H, d_h, r, "bf16", canary=True, groups=G)
    cache = PagedCache(*[dev(p, "bf16") for p in pools])
    L.append(dev(ac.X, "bf16"), dev(ac.positions, "i32"), dev(ac.seq_ids, "i32"),
             *[dev(getattr(w, n), "bf16") for n in ("W_S_K", "W_S_V", "U_K", "U_V")],
             cache, dev(ac.page_table, "i32"))
    f = lambda a: I.to_f64(a, "bf16")
    rows = grouped.project_grouped(f(ac.X), f(w.W_S_K), f(w.W_S_V), f(w.U_K), f(w.U_V), G)
    want = oracle.place([f(p) for p in pools], rows, ac.positions, ac.seq_ids, ac.page_table,
                        ac.page_size)
    for k, t in enumerate((cache.S_K, cache.S_V, cache.R_K, cache.R_V)):
        got = I.bf16_bits_to_f64(host_bits(t))
        np.testing.assert_array_equal(np.nan_to_num(got, nan=7.0), np.nan_to_num(want[k], nan=7.0))


def test_grouped_prefill_and_step():
    """Chunked prefill on a history and a decode step on a two-group cache
    (the per-row prefill and the separate append + decode run), against the
    oracle's decode over each row's visible keys."""
    import rank_kv_attention_gb300 as L
    from rank_kv_attention_gb300.api import PagedCache
    H, d_h, r, d, G = 16, 128, 48, 256, 2
    new, hist = [40, 90], [70, 5]
    caps = [a + b + 1 for a, b in zip(new, hist)]
    rng = np.random.default_rng(7)
    pt, num_pages = I.make_page_table(caps, 64, True, rng, 2)
    pools = I.empty_pools(num_pages, 64, H, d_h, r, "bf16", canary=True, groups=G)
    cache = PagedCache(*[dev(p, "bf16") for p in pools])
    w = I.make_weights(d, H, d_h, r, "bf16", seed=8, groups=G)
    Wd = [dev(getattr(w, n), "bf16") for n in ("W_S_K", "W_S_V", "U_K", "U_V")]
    draw = lambda n: I.f32_to_bf16_bits(rng.standard_normal((n, d)).astype(np.float32))
    Xh, Xn = draw(sum(hist)), draw(sum(new))
    Q = I.f32_to_bf16_bits(rng.standard_normal((sum(new), H, d_h)).astype(np.float32))
    pos_h = np.concatenate([np.arange(k) for k in hist]).astype(np.int32)
    sid_h = np.concatenate([np.full(k, b) for b, k in enumerate(hist)]).astype(np.int32)
    L.append(dev(Xh, "bf16"), dev(pos_h, "i32"), dev(sid_h, "i32"), *Wd, cache, dev(pt, "i32"))
    cu = np.array([0, new[0], sum(new)], np.int32)
    out = L.prefill(dev(Xn, "bf16"), dev(Q, "bf16"), dev(cu, "i32"), dev(np.array(hist, np.int32), "i32"),
                    int(max(caps)), *Wd, dev(w.B_K, "bf16"), dev(w.B_V, "bf16"), cache, dev(pt, "i32"))
    stored = [I.to_f64(host_bits(t), "bf16") for t in (cache.S_K, cache.S_V, cache.R_K, cache.R_V)]
    f = lambda a: I.to_f64(a, "bf16")
    pos_n = np.concatenate([np.arange(hist[b], hist[b] + new[b]) for b in range(2)])
    sid_n = np.concatenate([np.full(new[b], b) for b in range(2)])
    ref = grouped.decode_grouped(f(Q), *stored, f(w.B_K), f(w.B_V), pt[sid_n], pos_n + 1, 64)
    assert_close(host(out, "bf16"), ref, "bf16", "grouped prefill")
    # one decode step: append each request's next row and decode it
    Xs = draw(2)
    q = I.f32_to_bf16_bits(rng.standard_normal((2, H, d_h)).astype(np.float32))
    lens = np.array([hist[0] + new[0] + 1, hist[1] + new[1] + 1], np.int32)
    o = L.decode_step(dev(Xs, "bf16"), *Wd, dev(q, "bf16"), cache, dev(w.B_K, "bf16"), dev(w.B_V, "bf16"),
                      dev(lens, "i32"), dev(pt, "i32"), int(max(caps)))
    stored = [I.to_f64(host_bits(t), "bf16") for t in (cache.S_K, cache.S_V, cache.R_K, cache.R_V)]
    ref = grouped.decode_grouped(f(q), *stored, f(w.B_K), f(w.B_V), pt, lens, 64)
    assert_close(host(o, "bf16"), ref, "bf16", "grouped decode step")


def test_grouped_rope_and_norms():
    """The rotary embedding and the joint key norms with two groups: each
    group's heads against the single-basis oracles over that group's shared
    rows."""
    import rank_kv_attention_gb300 as L
    H, d_h, r, G = 16, 128, 48, 2
    lens = [300, 129, 77, 16]
    case = I.make_decode_case(4, H, d_h, r, lens, dtype="bf16", seed=12, shuffle=True, groups=G)
    dc = DevDecode(case)
    f = lambda a: I.to_f64(a, "bf16")
    SK, SV, RK, RV = pools_f64(case)
    hg = H // G
    table = L.rope_table(d_h, 300)
    got = host(L.decode_rope(dc.q, dc.cache, dc.B_K, dc.B_V, dc.seq_lens, dc.page_table, 300, table),
               "bf16")
    ref = np.empty_like(got)
    for g in range(G):
        hs = slice(g * hg, (g + 1) * hg)
        ref[:, hs] = R.decode_rope(f(case.q)[:, hs], SK[:, :, g], SV[:, :, g], RK[:, :, hs], RV[:, :, hs],
                                   f(case.B_K)[hs], f(case.B_V)[hs], case.page_table, case.seq_lens,
                                   case.page_size)
    assert_close(got, ref, "bf16", "grouped rope")
    # joint key norms of every cached row, then a normalised decode
    from rank_kv_attention_gb300.api import PagedCache
    eps = 1e-6
    NK = torch.zeros((case.num_pages, case.page_size, H), dtype=torch.bfloat16, device="cuda")
    cache = PagedCache(dc.cache.S_K, dc.cache.S_V, dc.cache.R_K, dc.cache.R_V, N_K=NK, norm_eps=eps)
    pos = np.concatenate([np.arange(L_) for L_ in lens]).astype(np.int32)
    sid = np.concatenate([np.full(L_, b) for b, L_ in enumerate(lens)]).astype(np.int32)
    L.key_norms(dev(pos, "i32"), dev(sid, "i32"), dc.B_K, cache, dc.page_table)
    got_nk = host(NK, "bf16")
    for b, L_ in enumerate(lens):
        rows = [oracle.gather_rows(p, case.page_table[b], L_, case.page_size) for p in (SK, RK)]
        for g in range(G):
            hs = slice(g * hg, (g + 1) * hg)
            want = N.key_norms(rows[0][:, g], rows[1][:, hs], f(case.B_K)[hs], eps)
            have = np.stack([got_nk[case.page_table[b, t // case.page_size], t % case.page_size, hs]
                             for t in range(L_)])
            np.testing.assert_allclose(have, want, rtol=1e-2, atol=1e-3)
    out = host(L.decode(dc.q, cache, dc.B_K, dc.B_V, dc.seq_lens, dc.page_table, 300), "bf16")
    ref = np.empty_like(out)
    for g in range(G):
        hs = slice(g * hg, (g + 1) * hg)
        ref[:, hs] = N.decode_norm(f(case.q)[:, hs], SK[:, :, g], SV[:, :, g], RK[:, :, hs], RV[:, :, hs],
                                   f(case.B_K)[hs], f(case.B_V)[hs], got_nk[:, :, hs], case.page_table,
                                   case.seq_lens, case.page_size)
    assert_close(out, ref, "bf16", "grouped norms")
