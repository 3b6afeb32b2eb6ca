"""GPU parity of lrkv_append (through the C ABI): bit-exact placement into
shuffled pages with canaries left untouched, bit-exact values when the
projections are exactly representable, float tolerance otherwise."""
import numpy as np
import pytest
import torch

import lrkv_inputs as I
import oracle
from gpu_util import assert_close, dev, host, host_bits

pytestmark = pytest.mark.gpu


def _run_append(ac, w, H, d_h, r, dtype, status=None):
    import rank_kv_attention_gb300 as L
    from rank_kv_attention_gb300.api import PagedCache
    pools = I.empty_pools(ac.num_pages, ac.page_size, H, d_h, r, dtype, canary=True)
    cache = PagedCache(*[dev(p, dtype) for p in pools])
    L.append(dev(ac.X, dtype), dev(ac.positions, "i32"), dev(ac.seq_ids, "i32"),
             dev(w.W_S_K, dtype), dev(w.W_S_V, dtype), dev(w.U_K, dtype), dev(w.U_V, dtype),
             cache, dev(ac.page_table, "i32"), status=status)
    return pools, cache


def _oracle_pools(ac, w, pools, dtype):
    f = lambda a: I.to_f64(a, dtype)
    rows = oracle.project(f(ac.X), f(w.W_S_K), f(w.W_S_V), f(w.U_K), f(w.U_V))
    return oracle.place([f(p) for p in pools], rows, ac.positions, ac.seq_ids, ac.page_table,
                        ac.page_size)


def _touched(ac):
    t = np.zeros((ac.num_pages, ac.page_size), bool)
    for b, p in zip(ac.seq_ids, ac.positions):
        t[ac.page_table[b, p // ac.page_size], p % ac.page_size] = True
    return t


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_append_exact_values_and_placement(dtype):
    """Integer-valued X and {-1,0,1} weights: every projection is a small
    integer, exact in fp32 accumulation and in bf16 storage, so the written
    bytes must equal the oracle's bit for bit, and untouched slots keep the
    canary."""
    H, d_h, r, d = 16, 128, 48, 256
    ac = I.make_append_case([37, 1, 130, 64], [0, 500, 63, 64], d, dtype=dtype, seed=1,
                            shuffle=True, spare_pages=2, interleave=True)
    rng = np.random.default_rng(2)
    Xi = rng.integers(-3, 4, size=ac.X.shape).astype(np.float32)
    ac.X = I.f32_to_bf16_bits(Xi) if dtype == "bf16" else Xi
    w = I.make_weights(d, H, d_h, r, dtype, seed=3)
    for name in ("W_S_K", "W_S_V", "U_K", "U_V"):
        a = getattr(w, name)
        vals = rng.integers(-1, 2, size=a.shape).astype(np.float32) * (rng.random(a.shape) < 0.1)
        setattr(w, name, I.f32_to_bf16_bits(vals) if dtype == "bf16" else vals.astype(np.float32))
    pools, cache = _run_append(ac, w, H, d_h, r, dtype)
    want = _oracle_pools(ac, w, pools, dtype)
    touched = _touched(ac)
    for k, t in enumerate((cache.S_K, cache.S_V, cache.R_K, cache.R_V)):
        got_bits = host_bits(t)
        if dtype == "bf16":
            want_bits = I.f32_to_bf16_bits(want[k].astype(np.float32))
        else:
            want_bits = want[k].astype(np.float32).view(np.uint32)
        assert np.array_equal(got_bits[touched], want_bits[touched]), f"pool {k}"
        canary = np.asarray(pools[k]).view(got_bits.dtype)
        assert np.array_equal(got_bits[~touched], canary[~touched]), f"pool {k} canary"


@pytest.mark.parametrize("H,d_h,r,d,dtype", [(16, 128, 48, 2048, "bf16"), (32, 128, 32, 512, "bf16"),
                                              (4, 16, 4, 64, "f32"), (8, 64, 24, 136, "bf16"),
                                              (8, 64, 24, 192, "bf16")])
def test_append_random_values(H, d_h, r, d, dtype):
    ac = I.make_append_case([100, 3, 77], [10, 0, 200], d, dtype=dtype, seed=H + r,
                            shuffle=True, interleave=True)
    w = I.make_weights(d, H, d_h, r, dtype, seed=4)
    pools, cache = _run_append(ac, w, H, d_h, r, dtype)
    want = _oracle_pools(ac, w, pools, dtype)
    touched = _touched(ac)
    for k, t in enumerate((cache.S_K, cache.S_V, cache.R_K, cache.R_V)):
        got = host(t, dtype)
        assert_close(got[touched], want[k][touched], dtype, f"pool {k}")
        assert np.all(np.isnan(got[~touched]))


def test_append_decode_step_rows():
    """The decode-step shape: one new row per request (B = 16, d = 2048)."""
    H, d_h, r, d = 16, 128, 48, 2048
    ac = I.make_append_case([1] * 16, list(range(4095, 4095 + 16)), d, seed=5, shuffle=True)
    w = I.make_weights(d, H, d_h, r, "bf16", seed=6)
    pools, cache = _run_append(ac, w, H, d_h, r, "bf16")
    want = _oracle_pools(ac, w, pools, "bf16")
    touched = _touched(ac)
    for k, t in enumerate((cache.S_K, cache.S_V, cache.R_K, cache.R_V)):
        assert_close(host(t, "bf16")[touched], want[k][touched], "bf16", f"pool {k}")


def test_append_bad_rows_skipped_and_flagged():
    import rank_kv_attention_gb300 as L
    H, d_h, r, d = 16, 128, 48, 64
    ac = I.make_append_case([5, 5], [0, 0], d, seed=7, shuffle=True, spare_pages=1)
    ac.seq_ids[1] = 7           # no such request
    ac.positions[2] = 10 ** 6   # beyond the page table
    ac.page_table[1, 0] = -5    # request 1's page is invalid
    w = I.make_weights(d, H, d_h, r, "bf16", seed=8)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pools, cache = _run_append(ac, w, H, d_h, r, "bf16", status=status)
    st = int(status.item())
    assert st & L.LRKV_STATUS_BAD_ROW and st & L.LRKV_STATUS_BAD_PAGE
    # only request 0's valid rows were written
    ok = [i for i in range(len(ac.positions))
          if ac.seq_ids[i] == 0 and ac.positions[i] < 10 ** 6]
    t = np.zeros((ac.num_pages, ac.page_size), bool)
    for i in ok:
        t[ac.page_table[0, ac.positions[i] // 64], ac.positions[i] % 64] = True
    got = host_bits(cache.S_K)
    assert np.all(got[~t] == I.BF16_NAN_BITS)
    assert not np.any(got[t] == I.BF16_NAN_BITS)


def _integer_case(n_per_seq, d, density, seed, H=16, d_h=128, r=48):
    """Integer rows in [-2, 2] and sparse {-1, 0, 1} weights: every projection
    is an integer of magnitude below 256, exact in fp32 accumulation and in
    bf16 storage, so the written bytes are fixed bit for bit."""
    ac = I.make_append_case(n_per_seq, [0] * len(n_per_seq), d, dtype="bf16", seed=seed,
                            shuffle=True, spare_pages=3, interleave=True)
    rng = np.random.default_rng(seed + 1)
    ac.X = I.f32_to_bf16_bits(rng.integers(-2, 3, size=ac.X.shape).astype(np.float32))
    w = I.make_weights(d, H, d_h, r, "bf16", seed=seed + 2)
    for name in ("W_S_K", "W_S_V", "U_K", "U_V"):
        a = getattr(w, name)
        vals = rng.integers(-1, 2, size=a.shape).astype(np.float32) * (rng.random(a.shape) < density)
        setattr(w, name, I.f32_to_bf16_bits(vals))
    return ac, w


# The persistent tensor-core projection walks its 128 x 256 output tiles with
# a stride of one grid (one CTA per SM); more than two grids' worth of tiles
# makes every CTA run its tile loop at least twice, so the second tensor-
# memory accumulator, the operand ring running on across tiles and the
# epilogue overlapping the next tile's products are all compared here.
@pytest.mark.parametrize("n_per_seq,d,density", [
    ([4096, 3000, 1173], 256, 0.1),   # 8269 rows: 65 x 7 = 455 tiles of 4 k-blocks
    ([3000, 2600], 2048, 0.02),       # 5600 rows at d = 2048: 44 x 7 = 308 tiles of 32 k-blocks
])
def test_append_many_tiles_bit_exact(n_per_seq, d, density):
    H, d_h, r = 16, 128, 48
    n = sum(n_per_seq)
    tiles = -(-n // 128) * ((2 * d_h + 2 * H * r) // 256)
    assert tiles > 2 * torch.cuda.get_device_properties(0).multi_processor_count
    ac, w = _integer_case(n_per_seq, d, density, seed=n % 1000)
    pools, cache = _run_append(ac, w, H, d_h, r, "bf16")
    want = _oracle_pools(ac, w, pools, "bf16")
    touched = _touched(ac)
    for k, t in enumerate((cache.S_K, cache.S_V, cache.R_K, cache.R_V)):
        wk = want[k][touched]
        assert np.all(wk == np.round(wk)) and np.abs(wk).max() < 256, "case must be exact in bf16"
        got_bits = host_bits(t)
        want_bits = I.f32_to_bf16_bits(want[k].astype(np.float32))
        assert np.array_equal(got_bits[touched], want_bits[touched]), f"pool {k}"
        canary = np.asarray(pools[k]).view(got_bits.dtype)
        assert np.array_equal(got_bits[~touched], canary[~touched]), f"pool {k} canary"
