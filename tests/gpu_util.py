"""Helpers shared by the GPU parity tests: moving seeded inputs to the device
and comparing the CUDA results with the float64 oracle.

Tolerances (written out here and in each test):
  * fp32 caches: max |got - ref| <= 1e-5 * max |ref| (normwise relative),
    and elementwise |got - ref| <= 1e-5 |ref| + 1e-6 max |ref| (relative
    error 1e-5 for every element, with a floor of a tenth of the normwise
    bound for elements that cancel to near zero, whose relative error no
    fp32 summation order can bound).
  * bf16 caches with fp32 accumulation: elementwise
    |got - ref| <= 2e-2 + 1e-2 |ref|, and additionally
    max |got - ref| <= 1e-2 * max |ref| (normwise), which bounds the error by
    a few bf16 output roundings (each <= 2^-9 relative) and catches a wrong
    term even when outputs are much smaller than the absolute tolerance.
"""
import numpy as np
import torch

import lrkv_inputs as I


def dev(arr, dtype):
    """Seeded numpy array -> contiguous CUDA tensor ('bf16' bit patterns or 'f32')."""
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16)
    elif dtype == "fp8":
        t = torch.from_numpy(np.ascontiguousarray(arr, dtype=np.uint8)).view(torch.float8_e4m3fn)
    elif dtype == "f32":
        t = torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32))
    else:
        t = torch.from_numpy(np.ascontiguousarray(arr, dtype=np.int32))
    return t.cuda()


def host(t, dtype):
    """CUDA tensor -> numpy float64 (exact widening)."""
    t = t.detach().cpu().contiguous()
    if dtype == "bf16":
        return I.bf16_bits_to_f64(t.view(torch.int16).numpy().view(np.uint16))
    return t.numpy().astype(np.float64)


def host_bits(t):
    """Raw storage bits of a CUDA tensor (uint16 for bf16, uint32 for fp32)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.view(torch.int32).numpy().view(np.uint32)


def assert_close(got, ref, dtype, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    if dtype == "f32":
        bound = 1e-5 * scale + 1e-30
        assert err.max(initial=0.0) <= bound, f"{what}: max err {err.max():.3e} > {bound:.3e}"
        ok = err <= 1e-5 * np.abs(ref) + 1e-6 * scale + 1e-30
        assert ok.all(), (f"{what}: {np.count_nonzero(~ok)} elements outside "
                          f"1e-5|ref| + 1e-6 max|ref| (worst {(err / (np.abs(ref) + 0.1 * scale + 1e-30)).max():.3e})")
    else:
        ok = err <= 2e-2 + 1e-2 * np.abs(ref)
        assert ok.all(), f"{what}: {np.count_nonzero(~ok)} elements outside 2e-2 + 1e-2|ref|"
        bound = 1e-2 * scale
        assert err.max(initial=0.0) <= bound, f"{what}: normwise err {err.max():.3e} > {bound:.3e}"
    return float(err.max(initial=0.0)), scale


class DevDecode:
    """A DecodeCase on the device plus a PagedCache over it."""

    def __init__(self, case):
        from rank_kv_attention_gb300.api import PagedCache
        dt, adt = case.dtype, case.act_dtype
        self.case = case
        self.q = dev(case.q, adt)
        self.cache = PagedCache(dev(case.S_K, dt), dev(case.S_V, dt), dev(case.R_K, dt),
                                dev(case.R_V, dt), tuple(case.scale))
        self.B_K = dev(case.B_K, adt)
        self.B_V = dev(case.B_V, adt)
        self.seq_lens = dev(case.seq_lens, "i32")
        self.page_table = dev(case.page_table, "i32")
        self.max_seq_len = int(max(1, case.seq_lens.max()))

    def run(self, status=None, out=None, ws=None):
        import rank_kv_attention_gb300 as L
        return L.decode(self.q, self.cache, self.B_K, self.B_V, self.seq_lens, self.page_table,
                        self.max_seq_len, out=out, ws=ws, status=status)


def pools_f64(case, pools=None):
    """float64 values of the four cache pools (8-bit codes times their scales)."""
    import oracle
    pools = pools if pools is not None else (case.S_K, case.S_V, case.R_K, case.R_V)
    if case.dtype == "fp8":
        return [oracle.fp8.dequantize(p, s) for p, s in zip(pools, case.scale)]
    return [I.to_f64(p, case.dtype) for p in pools]


def oracle_decode(case, pairs=None):
    import oracle
    f = lambda a: I.to_f64(a, case.act_dtype)
    fn = oracle.grouped.decode_grouped if case.groups > 1 else oracle.decode
    return fn(f(case.q), *pools_f64(case), f(case.B_K), f(case.B_V), case.page_table,
              case.seq_lens, case.page_size, pairs=pairs)
