"""GPU parity of lrkv_decode (called through the C ABI) against the float64
oracle, at small sizes over several tiles with ragged tails, and at the full
workload sizes on sampled (request, head) outputs."""
import numpy as np
import pytest
import torch

import lrkv_inputs as I
from gpu_util import DevDecode, assert_close, host, oracle_decode

pytestmark = pytest.mark.gpu

LENS = [1, 17, 300, 64, 65, 129]

# (H, d_h, r, dtype): the first group runs the tensor-core split kernel, the
# rest the generic kernel.
SHAPES = [
    (16, 128, 48, "bf16"), (16, 128, 56, "bf16"), (32, 128, 32, "bf16"), (16, 128, 32, "bf16"),
    (16, 128, 64, "bf16"), (16, 128, 16, "bf16"), (32, 128, 16, "bf16"),
    (8, 64, 24, "bf16"), (4, 128, 40, "bf16"), (4, 16, 4, "f32"), (6, 32, 8, "f32"),
]


@pytest.mark.parametrize("H,d_h,r,dtype", SHAPES)
def test_decode_small_parity(H, d_h, r, dtype):
    case = I.make_decode_case(len(LENS), H, d_h, r, LENS, dtype=dtype, seed=H * 1000 + r,
                              shuffle=True, spare_pages=3)
    got = host(DevDecode(case).run(), dtype)
    assert_close(got, oracle_decode(case), dtype, f"H={H} d_h={d_h} r={r}")


@pytest.mark.parametrize("page_size", [16, 32, 128])
def test_decode_page_sizes(page_size):
    case = I.make_decode_case(4, 16, 128, 48, [5, 33, 200, 16], seed=page_size, shuffle=True,
                              spare_pages=2, page_size=page_size)
    assert_close(host(DevDecode(case).run(), "bf16"), oracle_decode(case), "bf16")


@pytest.mark.parametrize("H,r", [(16, 48), (4, 40)])
def test_decode_tile_edges(H, r):
    lens = [1, 15, 16, 17, 63, 64, 65, 127, 128, 129, 1000]
    case = I.make_decode_case(len(lens), H, 128, r, lens, seed=3, shuffle=True)
    assert_close(host(DevDecode(case).run(), "bf16"), oracle_decode(case), "bf16")


def test_decode_single_long_request():
    case = I.make_decode_case(1, 16, 128, 48, [20000], seed=5)
    assert_close(host(DevDecode(case).run(), "bf16"), oracle_decode(case), "bf16")


def test_decode_many_short_requests():
    lens = np.random.default_rng(1).integers(1, 40, size=300)
    case = I.make_decode_case(len(lens), 16, 128, 56, lens, seed=6, shuffle=True)
    assert_close(host(DevDecode(case).run(), "bf16"), oracle_decode(case), "bf16")


def test_decode_zero_query_gives_mean_value():
    case = I.make_decode_case(2, 16, 128, 48, [50, 333], seed=7)
    case.q[:] = 0
    got = host(DevDecode(case).run(), "bf16")
    assert_close(got, oracle_decode(case), "bf16")


def test_decode_stale_workspace_and_determinism():
    case = I.make_decode_case(3, 32, 128, 32, [700, 5, 2500], seed=8, shuffle=True)
    d = DevDecode(case)
    import rank_kv_attention_gb300 as L
    ws = L.workspace(L.decode_workspace_bytes(3, 32, 128, 32, d.max_seq_len))
    ws.fill_(0xFF)
    a = d.run(ws=ws).clone()
    ws.fill_(0x7F)
    b = d.run(ws=ws)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert_close(host(a, "bf16"), oracle_decode(case), "bf16")


def test_decode_bad_metadata_is_flagged_not_read():
    import rank_kv_attention_gb300 as L
    lens = [40, 100, 70]
    case = I.make_decode_case(3, 16, 128, 48, lens, seed=9, shuffle=True, spare_pages=1)
    d = DevDecode(case)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    # request 0: length 0 (invalid); request 2: a page id outside the pool
    d.seq_lens[0] = 0
    d.page_table[2, 1] = 10 ** 6
    out = host(d.run(status=status), "bf16")
    st = int(status.item())
    assert st & L.LRKV_STATUS_BAD_SEQLEN and st & L.LRKV_STATUS_BAD_PAGE
    assert np.all(out[0] == 0)
    assert np.all(np.isfinite(out))
    # the untouched request still matches
    ref = oracle_decode(case, pairs=[(1, h) for h in range(16)])
    assert_close(out[1], ref[1], "bf16")


# --------------------------------------------------------------------------
# Full workload sizes
# --------------------------------------------------------------------------
def _pairs(B, H, k, seed):
    rng = np.random.default_rng(seed)
    pairs = {(b, int(rng.integers(H))) for b in range(B)}
    while len(pairs) < k:
        pairs.add((int(rng.integers(B)), int(rng.integers(H))))
    return sorted(pairs)


def test_decode_T4096_full():
    case = I.config_decode_case("decode_T4096")
    got = host(DevDecode(case).run(), "bf16")
    assert_close(got, oracle_decode(case), "bf16", "B=16 H=16 r=48 T=4096")


def test_decode_T32768_sampled():
    case = I.config_decode_case("decode_T32768")
    got = host(DevDecode(case).run(), "bf16")
    pairs = _pairs(case.B, case.H, 16, 11)
    ref = oracle_decode(case, pairs)
    idx = tuple(np.array(pairs).T)
    assert_close(got[idx], ref[idx], "bf16", "B=4 H=32 r=32 T=32768")
    assert np.all(np.isfinite(got))


def test_decode_ragged_paged_sampled():
    case = I.config_decode_case("ragged_paged")
    got = host(DevDecode(case).run(), "bf16")
    pairs = _pairs(case.B, case.H, 96, 12)
    ref = oracle_decode(case, pairs)
    idx = tuple(np.array(pairs).T)
    assert_close(got[idx], ref[idx], "bf16", "ragged B=64 H=16 r=56")
    assert np.all(np.isfinite(got))
