"""GPU parity of the exact rotary embedding (reading note "Low-Rank Key Value
Attention", section 8) through the C ABI, against the float64 oracle: the
cos/sin table, decode over bf16, fp32 and 8-bit caches (ranges that cut
requests mid-way, so a segment's query lies beyond it), a query beyond the
table, chunked prefill on a history, and the 16 x 4096 workload sampled."""
import numpy as np
import pytest
import torch

import lrkv_inputs as I
import oracle
from oracle import rope as R
from gpu_util import DevDecode, assert_close, dev, host, host_bits, pools_f64

pytestmark = pytest.mark.gpu


def test_rope_table_values():
    import rank_kv_attention_gb300 as L
    for d_h, n in ((128, 5000), (16, 70), (2, 3)):
        tab = L.rope_table(d_h, n)
        t = tab.cos_sin.cpu().numpy().astype(np.float64)
        ref = R.table(d_h, n)
        # one rounding of a value in [-1, 1] to float: <= 2^-25 (2^-24 at 1)
        assert np.abs(t - ref).max() <= 6e-8, (d_h, np.abs(t - ref).max())
        # the f16 copy: one round-to-nearest-even of the double value, the
        # same rounding numpy applies from float64
        t16 = tab.cos_sin_f16.cpu().numpy()
        assert np.array_equal(t16.view(np.uint16), ref.astype(np.float16).view(np.uint16)), d_h


def _oracle_rope(case, pairs=None):
    f = lambda a: I.to_f64(a, case.act_dtype)
    return R.decode_rope(f(case.q), *pools_f64(case), f(case.B_K), f(case.B_V), case.page_table,
                         case.seq_lens, case.page_size, pairs=pairs)


def _run_rope(case, table, status=None):
    import rank_kv_attention_gb300 as L
    dc = DevDecode(case)
    return L.decode_rope(dc.q, dc.cache, dc.B_K, dc.B_V, dc.seq_lens, dc.page_table, dc.max_seq_len,
                         table, status=status)


LENS = [1, 2, 17, 300, 64, 65, 129, 900]


# the tensor-core rotary kernel at every group shape: 4 heads with 128-byte
# (r = 48, 32, 16) or 64-byte (r = 56, one R_K buffer) swizzled R_K, 2 heads
# (r = 64), H = 32, and pages of 32, 64 and 128 rows
@pytest.mark.parametrize("H,d_h,r,dtype,ps", [(16, 128, 48, "bf16", 64), (8, 64, 24, "bf16", 16),
                                              (4, 16, 4, "f32", 64), (32, 128, 32, "bf16", 32),
                                              (16, 128, 64, "bf16", 64), (16, 128, 56, "fp8", 64),
                                              (2, 256, 8, "f32", 16), (16, 128, 56, "bf16", 64),
                                              (16, 128, 16, "bf16", 128), (16, 128, 32, "bf16", 32)])
def test_rope_decode_parity(H, d_h, r, dtype, ps):
    import rank_kv_attention_gb300 as L
    case = I.make_decode_case(len(LENS), H, d_h, r, LENS, dtype=dtype, seed=H + r, shuffle=True,
                              spare_pages=2, page_size=ps)
    table = L.rope_table(d_h, int(case.seq_lens.max()))
    got = host(_run_rope(case, table), case.act_dtype)
    assert_close(got, _oracle_rope(case), case.act_dtype, f"rope H={H} d_h={d_h} r={r} {dtype}")


def test_rope_long_request_cut_into_segments():
    """One 6000-row request among short ones: the plan cuts it across many
    CTAs, and every segment must use the request's last position for the
    query."""
    import rank_kv_attention_gb300 as L
    lens = [6000, 3, 40]
    case = I.make_decode_case(3, 16, 128, 48, lens, dtype="bf16", seed=3, shuffle=True)
    table = L.rope_table(128, 6000)
    got = host(_run_rope(case, table), "bf16")
    pairs = [(0, h) for h in range(0, 16, 3)] + [(1, 0), (2, 5)]
    ref = _oracle_rope(case, pairs)
    idx = tuple(np.array(pairs).T)
    assert_close(got[idx], ref[idx], "bf16", "long request")


def test_rope_query_beyond_table():
    """A request longer than the table covers (allowed by the page table) is
    not attended: zero output and LRKV_STATUS_BAD_SEQLEN; the others are
    unaffected."""
    import rank_kv_attention_gb300 as L
    lens = [100, 200, 50]
    case = I.make_decode_case(3, 16, 128, 48, lens, dtype="bf16", seed=4, spare_pages=1)
    dc = DevDecode(case)
    table = L.rope_table(128, 150)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = L.decode_rope(dc.q, dc.cache, dc.B_K, dc.B_V, dc.seq_lens, dc.page_table, 150, table,
                        status=st)
    assert int(st.item()) & L.LRKV_STATUS_BAD_SEQLEN
    got = host(out, "bf16")
    assert np.all(got[1] == 0)
    ref = _oracle_rope(case, [(b, h) for b in (0, 2) for h in range(16)])
    assert_close(got[[0, 2]], ref[[0, 2]], "bf16", "valid requests")


def test_rope_prefill_chunk_on_history():
    """Chunked prefill with the rotary embedding: every new row (query at its
    own position) attends its request's rows up to that position."""
    import rank_kv_attention_gb300 as L
    from rank_kv_attention_gb300.api import PagedCache
    H, d_h, r, d = 16, 128, 48, 256
    new, hist = [40, 90], [70, 5]
    caps = [a + b for a, b in zip(new, hist)]
    rng = np.random.default_rng(7)
    pt, num_pages = I.make_page_table(caps, 64, True, rng, 2)
    pools = I.empty_pools(num_pages, 64, H, d_h, r, "bf16", canary=True)
    cache = PagedCache(*[dev(p, "bf16") for p in pools])
    w = I.make_weights(d, H, d_h, r, "bf16", seed=8)
    draw = lambda n: I.f32_to_bf16_bits(rng.standard_normal((n, d)).astype(np.float32))
    Xh, Xn = draw(sum(hist)), draw(sum(new))
    Q = I.f32_to_bf16_bits(rng.standard_normal((sum(new), H, d_h)).astype(np.float32))
    pos_h = np.concatenate([np.arange(k) for k in hist]).astype(np.int32)
    sid_h = np.concatenate([np.full(k, b) for b, k in enumerate(hist)]).astype(np.int32)
    Wd = [dev(getattr(w, n), "bf16") for n in ("W_S_K", "W_S_V", "U_K", "U_V")]
    L.append(dev(Xh, "bf16"), dev(pos_h, "i32"), dev(sid_h, "i32"), *Wd, cache, dev(pt, "i32"))
    table = L.rope_table(d_h, int(max(caps)))
    cu = np.array([0, new[0], sum(new)], np.int32)
    out = L.prefill_rope(dev(Xn, "bf16"), dev(Q, "bf16"), dev(cu, "i32"),
                         dev(np.array(hist, np.int32), "i32"), int(max(caps)), *Wd,
                         dev(w.B_K, "bf16"), dev(w.B_V, "bf16"), cache, dev(pt, "i32"), table)
    stored = [I.to_f64(host_bits(t), "bf16") for t in (cache.S_K, cache.S_V, cache.R_K, cache.R_V)]
    f = lambda a: I.to_f64(a, "bf16")
    pos_n = np.concatenate([np.arange(hist[b], hist[b] + new[b]) for b in range(2)])
    sid_n = np.concatenate([np.full(new[b], b) for b in range(2)])
    ref = R.decode_rope(f(Q), *stored, f(w.B_K), f(w.B_V), pt[sid_n], pos_n + 1, 64)
    assert_close(host(out, "bf16"), ref, "bf16", "rope prefill")


def test_rope_T4096_sampled():
    """The 16 x 4096 decode workload with the rotary embedding, sampled."""
    import rank_kv_attention_gb300 as L
    case = I.config_decode_case("decode_T4096")
    table = L.rope_table(128, 4096)
    got = host(_run_rope(case, table), "bf16")
    rng = np.random.default_rng(9)
    pairs = sorted({(b, int(rng.integers(case.H))) for b in range(0, case.B, 3)} | {(15, 15)})
    ref = _oracle_rope(case, pairs)
    idx = tuple(np.array(pairs).T)
    assert_close(got[idx], ref[idx], "bf16", "decode_T4096 rope")


def test_rope_many_requests_in_one_range():
    """More requests inside one CTA's rows than its local offset table holds
    (zero-length requests in between): the score and split kernels take the
    prologue's offsets; the invalid lengths get zero and a flag."""
    import rank_kv_attention_gb300 as L
    lens = [0] * 100 + [40] + [0] * 100 + [23]
    case = I.make_decode_case(len(lens), 16, 128, 48, lens, dtype="bf16", seed=11, shuffle=True)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    table = L.rope_table(128, 64)
    got = host(_run_rope(case, table, status=st), "bf16")
    assert int(st.item()) & L.LRKV_STATUS_BAD_SEQLEN
    valid = [100, 201]
    assert np.all(np.delete(got, valid, axis=0) == 0)
    ref = _oracle_rope(case, [(b, h) for b in valid for h in range(16)])
    assert_close(got[valid], ref[valid], "bf16", "requests among empty ones")


def test_rope_stale_workspace_and_length_bound():
    """The tensor-core rotary path writes every score it reads (a workspace
    full of stale bytes gives the same bits), and on it a request longer than
    max_seq_len is not attended (zero output, LRKV_STATUS_BAD_SEQLEN)."""
    import rank_kv_attention_gb300 as L
    lens = [300, 129, 77, 16]
    case = I.make_decode_case(4, 16, 128, 48, lens, dtype="bf16", seed=12, shuffle=True)
    dc = DevDecode(case)
    table = L.rope_table(128, 300)
    ws = L.workspace(L.decode_rope_workspace_bytes(4, 16, 128, 48, 300))
    runs = []
    for fill in (0xFF, 0x7F):
        ws.fill_(fill)
        runs.append(L.decode_rope(dc.q, dc.cache, dc.B_K, dc.B_V, dc.seq_lens, dc.page_table, 300,
                                  table, ws=ws).clone())
    assert torch.equal(runs[0].view(torch.int16), runs[1].view(torch.int16))
    assert_close(host(runs[0], "bf16"), _oracle_rope(case), "bf16", "stale workspace")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = host(L.decode_rope(dc.q, dc.cache, dc.B_K, dc.B_V, dc.seq_lens, dc.page_table, 200,
                             table, status=st), "bf16")
    assert int(st.item()) & L.LRKV_STATUS_BAD_SEQLEN
    assert np.all(out[0] == 0)
    ref = _oracle_rope(case, [(b, h) for b in (1, 2, 3) for h in range(16)])
    assert_close(out[1:], ref[1:], "bf16", "requests within max_seq_len")
