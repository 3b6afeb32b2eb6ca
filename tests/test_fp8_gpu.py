"""GPU parity of the 8-bit (E4M3) cache through the C ABI: decode against the
float64 oracle over the dequantized pools; append writes the codes the
oracle's encoder gives (bit-exact when the projections are exact, at most one
code step apart at rounding boundaries otherwise) and leaves every other slot
untouched; prefill and the decode step attend over the quantized rows."""
import numpy as np
import pytest
import torch

import lrkv_inputs as I
import oracle
from gpu_util import DevDecode, assert_close, dev, host, host_bits, oracle_decode

pytestmark = pytest.mark.gpu

LENS = [1, 17, 300, 64, 65, 129]


@pytest.mark.parametrize("H,d_h,r", [(16, 128, 48), (32, 128, 32), (16, 128, 56), (8, 64, 24),
                                     (4, 128, 40), (16, 128, 16)])
def test_fp8_decode_parity(H, d_h, r):
    case = I.make_decode_case(len(LENS), H, d_h, r, LENS, dtype="fp8", seed=H + r + d_h,
                              shuffle=True, spare_pages=3)
    got = host(DevDecode(case).run(), "bf16")
    assert_close(got, oracle_decode(case), "bf16", f"fp8 H={H} d_h={d_h} r={r}")


def test_fp8_decode_page_sizes_and_long():
    for ps, lens in ((32, [5, 33, 200, 16]), (128, [300, 1, 1000]), (64, [5000])):
        case = I.make_decode_case(len(lens), 16, 128, 48, lens, dtype="fp8", seed=ps,
                                  shuffle=True, spare_pages=2, page_size=ps)
        assert_close(host(DevDecode(case).run(), "bf16"), oracle_decode(case), "bf16", f"ps={ps}")


@pytest.mark.parametrize("H,r", [(16, 48), (32, 32), (16, 56)])
@pytest.mark.parametrize("q_scale", [2.0 ** 20, 2.0 ** -20])
def test_fp8_decode_query_range(H, r, q_scale):
    """Queries far outside f16 range (and tiny ones), with the cache values
    scaled the other way so the scores stay ordinary: the tensor-core kernel
    rescales q and p per head by a power of two before rounding them to f16."""
    case = I.make_decode_case(4, H, 128, r, [700, 33, 1, 260], dtype="fp8", seed=5, shuffle=True,
                              q_std=q_scale, cache_std=1.0 / q_scale,
                              fp8_scale=I.FP8_SCALE / q_scale)
    got = host(DevDecode(case).run(), "bf16")
    assert np.all(np.isfinite(got))
    # outputs scale with the cache (1 / q_scale); compare at unit scale, where
    # the tolerance's absolute term means what it does elsewhere (power-of-two
    # scaling is exact on both sides)
    assert_close(got * q_scale, oracle_decode(case) * q_scale, "bf16", f"q x {q_scale}")


@pytest.mark.parametrize("scales", [(0.37, 1.3, 0.05, 2.1), (2.0 ** -9, 2.0 ** 3, 1.0, 0.01)])
def test_fp8_decode_pool_scales(scales):
    """Different, non-power-of-two scales per pool on the tensor-core shapes."""
    for H, r in ((16, 48), (32, 16)):
        case = I.make_decode_case(5, H, 128, r, [129, 1000, 17, 64, 5], dtype="fp8", seed=H + r,
                                  shuffle=True, spare_pages=1, fp8_scale=scales)
        assert_close(host(DevDecode(case).run(), "bf16"), oracle_decode(case), "bf16",
                     f"H={H} r={r} scales={scales}")


def test_fp8_decode_T4096_sampled():
    """The 16 x 4096 decode workload over an 8-bit cache, on sampled
    (request, head) outputs."""
    case = I.config_decode_case("decode_T4096_fp8")
    got = host(DevDecode(case).run(), "bf16")
    rng = np.random.default_rng(3)
    pairs = sorted({(b, int(rng.integers(case.H))) for b in range(case.B)} | {(0, 0), (15, 15)})
    ref = oracle_decode(case, pairs=pairs)
    idx = tuple(np.array(pairs).T)
    assert_close(got[idx], ref[idx], "bf16", "decode_T4096_fp8")


def _append_fp8(X, w, ac, H, d_h, r, scales):
    import rank_kv_attention_gb300 as L
    from rank_kv_attention_gb300.api import PagedCache
    pools = I.empty_pools(ac.num_pages, ac.page_size, H, d_h, r, "fp8", canary=True)
    cache = PagedCache(*[dev(p, "fp8") for p in pools], tuple(scales))
    L.append(dev(X, "bf16"), dev(ac.positions, "i32"), dev(ac.seq_ids, "i32"),
             dev(w.W_S_K, "bf16"), dev(w.W_S_V, "bf16"), dev(w.U_K, "bf16"), dev(w.U_V, "bf16"),
             cache, dev(ac.page_table, "i32"))
    return pools, cache


def _assert_near_codes(got, want, what):
    """Codes from the kernel's fp32 projection and the oracle's float64 one:
    equal, or adjacent (one step apart in magnitude, same sign; +0 and -0
    count as adjacent) where the value sits at a rounding boundary, and
    rarely so."""
    g, o = np.asarray(got).astype(np.int64), np.asarray(want).astype(np.int64)
    same_sign = ((g ^ o) & 0x80) == 0
    step = np.where(same_sign, np.abs((g & 0x7F) - (o & 0x7F)),
                    (g & 0x7F) + (o & 0x7F) + 1)
    assert step.max(initial=0) <= 1, f"{what}: codes more than one step apart"
    assert (step > 0).mean() < 1e-3, f"{what}: {(step > 0).mean():.2e} of the codes differ"


def _touched(ac):
    t = np.zeros((ac.num_pages, ac.page_size), bool)
    for b, p in zip(ac.seq_ids, ac.positions):
        t[ac.page_table[b, p // ac.page_size], p % ac.page_size] = True
    return t


def _oracle_codes(X, w, ac, pools, scales):
    f = lambda a: I.to_f64(a, "bf16")
    rows = oracle.project(f(X), f(w.W_S_K), f(w.W_S_V), f(w.U_K), f(w.U_V))
    codes = [oracle.fp8.quantize(x, s) for x, s in zip(rows, scales)]
    return oracle.place([np.array(p) for p in pools], codes, ac.positions, ac.seq_ids,
                        ac.page_table, ac.page_size)


@pytest.mark.parametrize("n_per_seq,start", [([37, 1, 130, 64], [0, 500, 63, 64]),
                                             ([1] * 16, list(range(4095, 4095 + 16)))])
def test_fp8_append_exact_codes(n_per_seq, start):
    """Integer X and sparse {-1, 0, 1} weights: every projection is an exact
    integer in both fp32 and float64, so both sides round the same value and
    the written codes must be identical; other slots keep the canary."""
    H, d_h, r, d = 16, 128, 48, 256
    scales = (1.0, 0.5, 2.0, 0.25)
    ac = I.make_append_case(n_per_seq, start, d, dtype="bf16", seed=1, shuffle=True,
                            spare_pages=2, interleave=True)
    rng = np.random.default_rng(2)
    X = I.f32_to_bf16_bits(rng.integers(-3, 4, size=(len(ac.positions), d)).astype(np.float32))
    w = I.make_weights(d, H, d_h, r, "bf16", seed=3)
    for name in ("W_S_K", "W_S_V", "U_K", "U_V"):
        a = getattr(w, name)
        vals = rng.integers(-1, 2, size=a.shape).astype(np.float32) * (rng.random(a.shape) < 0.1)
        setattr(w, name, I.f32_to_bf16_bits(vals))
    pools, cache = _append_fp8(X, w, ac, H, d_h, r, scales)
    want = _oracle_codes(X, w, ac, pools, scales)
    for k, t in enumerate((cache.S_K, cache.S_V, cache.R_K, cache.R_V)):
        assert np.array_equal(host_bits(t), want[k]), f"pool {k}"


@pytest.mark.parametrize("n_per_seq,d", [([100, 3, 77], 2048), ([1] * 16, 2048), ([300], 512)])
def test_fp8_append_random_codes(n_per_seq, d):
    """Random rows: the kernel rounds its fp32 projection, the oracle its
    float64 one; they may land on adjacent codes only where the value sits at
    a rounding boundary."""
    H, d_h, r = 16, 128, 48
    scales = (2.0 ** -5,) * 4
    ac = I.make_append_case(n_per_seq, [10] * len(n_per_seq), d, dtype="bf16", seed=4,
                            shuffle=True, interleave=True)
    rng = np.random.default_rng(5)
    X = I.f32_to_bf16_bits(rng.standard_normal((len(ac.positions), d)).astype(np.float32))
    w = I.make_weights(d, H, d_h, r, "bf16", seed=6)
    pools, cache = _append_fp8(X, w, ac, H, d_h, r, scales)
    want = _oracle_codes(X, w, ac, pools, scales)
    touched = _touched(ac)
    for k, t in enumerate((cache.S_K, cache.S_V, cache.R_K, cache.R_V)):
        got = host_bits(t)
        assert np.array_equal(got[~touched], want[k][~touched]), f"pool {k} canary"
        _assert_near_codes(got[touched], want[k][touched], f"pool {k}")


def test_fp8_prefill_parity():
    """Chunked prefill onto an 8-bit cache: every new row attends over the
    quantized rows of its request up to its position."""
    import rank_kv_attention_gb300 as L
    from rank_kv_attention_gb300.api import PagedCache
    H, d_h, r, d = 16, 128, 48, 256
    scales = (2.0 ** -5,) * 4
    new, hist = [40, 90], [70, 5]
    caps = [a + b for a, b in zip(new, hist)]
    rng = np.random.default_rng(7)
    pt, num_pages = I.make_page_table(caps, 64, True, rng, 2)
    pools = I.empty_pools(num_pages, 64, H, d_h, r, "fp8", canary=True)
    cache = PagedCache(*[dev(p, "fp8") for p in pools], scales)
    w = I.make_weights(d, H, d_h, r, "bf16", seed=8)
    draw = lambda n: I.f32_to_bf16_bits(rng.standard_normal((n, d)).astype(np.float32))
    Xh, Xn = draw(sum(hist)), draw(sum(new))
    Q = I.f32_to_bf16_bits(rng.standard_normal((sum(new), H, d_h)).astype(np.float32))
    pos_h = np.concatenate([np.arange(k) for k in hist]).astype(np.int32)
    sid_h = np.concatenate([np.full(k, b) for b, k in enumerate(hist)]).astype(np.int32)
    Wd = [dev(getattr(w, n), "bf16") for n in ("W_S_K", "W_S_V", "U_K", "U_V")]
    L.append(dev(Xh, "bf16"), dev(pos_h, "i32"), dev(sid_h, "i32"), *Wd, cache, dev(pt, "i32"))
    cu = np.array([0, new[0], sum(new)], np.int32)
    out = L.prefill(dev(Xn, "bf16"), dev(Q, "bf16"), dev(cu, "i32"), dev(np.array(hist), "i32"),
                    int(max(caps)), *Wd, dev(w.B_K, "bf16"), dev(w.B_V, "bf16"), cache,
                    dev(pt, "i32"))
    # oracle: the cache the GPU wrote, decoded with the scales (its codes may
    # differ from the oracle's own rounding by one step at boundaries, and the
    # attention must use the stored values), then one decode per new row
    stored = [oracle.fp8.dequantize(host_bits(t), s)
              for t, s in zip((cache.S_K, cache.S_V, cache.R_K, cache.R_V), scales)]
    f = lambda a: I.to_f64(a, "bf16")
    pos_n = np.concatenate([np.arange(hist[b], hist[b] + new[b]) for b in range(2)])
    sid_n = np.concatenate([np.full(new[b], b) for b in range(2)])
    ref = oracle.decode(f(Q), *stored, f(w.B_K), f(w.B_V), pt[sid_n], pos_n + 1, 64)
    assert_close(host(out, "bf16"), ref, "bf16", "fp8 prefill")
    # and the stored new rows are the oracle's codes of its own projections
    rows = oracle.project(f(Xn), *[f(getattr(w, n)) for n in ("W_S_K", "W_S_V", "U_K", "U_V")])
    for k, (x, s) in enumerate(zip(rows, scales)):
        want = oracle.fp8.quantize(x, s)
        got = host_bits((cache.S_K, cache.S_V, cache.R_K, cache.R_V)[k])
        slots = [(pt[b, p // 64], p % 64) for b, p in zip(sid_n, pos_n)]
        _assert_near_codes(np.stack([got[a, c] for a, c in slots]), want, f"pool {k} new rows")


def test_fp8_decode_step():
    """lrkv_decode_step on an 8-bit cache (append, then decode): the new rows
    are stored as codes and attended."""
    import rank_kv_attention_gb300 as L
    lens = [1, 17, 300, 64]
    case = I.make_decode_case(len(lens), 16, 128, 48, lens, dtype="fp8", seed=9, shuffle=True,
                              spare_pages=2)
    w = I.make_weights(512, 16, 128, 48, "bf16", seed=10)
    X = I.f32_to_bf16_bits(np.random.default_rng(11).standard_normal((len(lens), 512))
                           .astype(np.float32))
    dc = DevDecode(case)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = L.decode_step(dev(X, "bf16"), *[dev(getattr(w, n), "bf16") for n in
                                          ("W_S_K", "W_S_V", "U_K", "U_V")],
                        dc.q, dc.cache, dc.B_K, dc.B_V, dc.seq_lens, dc.page_table,
                        dc.max_seq_len, status=st)
    assert int(st.item()) == 0
    pools = (dc.cache.S_K, dc.cache.S_V, dc.cache.R_K, dc.cache.R_V)
    stored = [oracle.fp8.dequantize(host_bits(t), s) for t, s in zip(pools, case.scale)]
    f = lambda a: I.to_f64(a, "bf16")
    # the new rows (position L - 1) hold the oracle's codes of its projections;
    # every other slot keeps its bytes
    rows = oracle.project(f(X), *[f(getattr(w, n)) for n in ("W_S_K", "W_S_V", "U_K", "U_V")])
    new = np.zeros((case.num_pages, case.page_size), bool)
    for b, L in enumerate(case.seq_lens):
        new[case.page_table[b, (L - 1) // case.page_size], (L - 1) % case.page_size] = True
    for k, (t, orig) in enumerate(zip(pools, (case.S_K, case.S_V, case.R_K, case.R_V))):
        got = host_bits(t)
        assert np.array_equal(got[~new], orig[~new]), f"pool {k} other slots"
        slots = [(case.page_table[b, (L - 1) // case.page_size], (L - 1) % case.page_size)
                 for b, L in enumerate(case.seq_lens)]
        _assert_near_codes(np.stack([got[a, c] for a, c in slots]),
                           oracle.fp8.quantize(rows[k], case.scale[k]), f"pool {k} new rows")
    ref = oracle.decode(f(case.q), *stored, f(case.B_K), f(case.B_V), case.page_table,
                        case.seq_lens, case.page_size)
    assert_close(host(out, "bf16"), ref, "bf16", "fp8 decode step")
