"""Seeded synthetic inputs for LRKV decode, append and prefill.

This module draws random tensors and lays them out; it holds none of the
attention arithmetic.  Both the float64 oracle (``oracle/``) and the CUDA path
(``rank_kv_attention_gb300``) receive the arrays made here, so their results
can be compared element by element.

Conventions (shared with the C-ABI in ``include/lrkv.h``):

* bf16 tensors are carried as ``uint16`` bit patterns.  ``f32_to_bf16_bits``
  rounds to nearest even; ``bf16_bits_to_f64`` widens exactly.
* Cache pools are paged with ``page_size`` tokens per page:
  ``S_K, S_V: [num_pages, page_size, d_h]`` and
  ``R_K, R_V: [num_pages, page_size, H, r]`` (token-major, all heads of one
  token contiguous).  The same page id indexes all four pools.
* ``page_table: [B, max_pages] int32``; entries past a request's last page
  are -1.  Slots past ``seq_len`` inside the last page hold a NaN canary.
* Projection weights are stored output-major (as ``nn.Linear.weight``):
  ``W_S_K, W_S_V: [d_h, d]`` and ``U_K, U_V: [H, r, d]``.  The per-head
  expansion bases keep the paper's orientation: ``B_K, B_V: [H, d_h, r]``.

Distributions follow the workloads of the LRKV reading note (Low-Rank Key
Value Attention, section 3 and the configurations it is measured on):
activations and weights ~ N(0, 1/d), expansion bases ~ N(0, 1/r), decode
queries and cache rows ~ N(0, 1).
"""
from __future__ import annotations

import dataclasses
import numpy as np

PAGE_SIZE = 64
BF16_NAN_BITS = np.uint16(0x7FC1)  # canary for never-written cache slots
F32_NAN_CANARY = np.float32(np.nan)
FP8_NAN_CODE = np.uint8(0x7F)      # the same for 8-bit (E4M3) pools
FP8_SCALE = 2.0 ** -5              # pool scale of the 8-bit cases: N(0,1) values use codes up to ~160


# ----------------------------------------------------------------------------
# bf16 encoding (storage format only)
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(x) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    out = ((u + bias) >> 16).astype(np.uint16)
    if nan.any():
        out[nan] = BF16_NAN_BITS
    return out


def bf16_bits_to_f32(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_bits_to_f64(b) -> np.ndarray:
    return bf16_bits_to_f32(b).astype(np.float64)


# ----------------------------------------------------------------------------
# 8-bit (E4M3) codes (storage format only; the values they stand for are
# defined by the oracle)
# ----------------------------------------------------------------------------
def f32_to_e4m3_codes(x) -> np.ndarray:
    """Codes of float32 values (torch's float8_e4m3fn conversion), clamped to
    the finite range first."""
    import torch
    v = np.clip(np.ascontiguousarray(x, dtype=np.float32), -448.0, 448.0)
    return torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def act_dtype(dtype: str) -> str:
    """Element type of the non-cache tensors used with a cache of this type."""
    return "bf16" if dtype == "fp8" else dtype


def to_f64(a, dtype: str) -> np.ndarray:
    """Exact float64 view of a stored tensor ('bf16' bits or 'f32')."""
    if dtype == "bf16":
        return bf16_bits_to_f64(a)
    return np.asarray(a, dtype=np.float32).astype(np.float64)


def _draw(rng: np.random.Generator, shape, std: float, dtype: str, scale: float = 1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if dtype == "fp8":
        return f32_to_e4m3_codes(x / np.float32(scale))
    return f32_to_bf16_bits(x) if dtype == "bf16" else x


def _draw_chunked(rng, shape, std, dtype, chunk_elems=1 << 24, scale=1.0):
    """Like _draw but bounds the float32 temporary for very large pools."""
    shape = tuple(int(s) for s in shape)
    lead = shape[0]
    inner = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    kind = {"bf16": np.uint16, "fp8": np.uint8}.get(dtype, np.float32)
    out = np.empty(shape, dtype=kind)
    flat = out.reshape(lead, inner)
    step = max(1, chunk_elems // max(1, inner))
    for s in range(0, lead, step):
        e = min(lead, s + step)
        flat[s:e] = _draw(rng, (e - s, inner), std, dtype, scale)
    return out


# ----------------------------------------------------------------------------
# Page tables
# ----------------------------------------------------------------------------
def make_page_table(seq_caps, page_size=PAGE_SIZE, shuffle=False, rng=None,
                    spare_pages=0, max_pages=None):
    """Assign pages to requests.

    ``seq_caps[b]`` is the number of token slots request b needs.  Pages are
    numbered 0..num_pages-1; with ``shuffle`` the ids are a random
    permutation of the pool (pages of one request scattered), else request b
    owns a contiguous run.  Returns (page_table [B, max_pages] int32,
    num_pages).
    """
    seq_caps = np.asarray(seq_caps, dtype=np.int64)
    n_pages_b = (seq_caps + page_size - 1) // page_size
    total = int(n_pages_b.sum())
    num_pages = total + int(spare_pages)
    if max_pages is None:
        max_pages = int(n_pages_b.max()) if len(n_pages_b) else 1
    max_pages = max(1, int(max_pages))
    ids = np.arange(num_pages, dtype=np.int64)
    if shuffle:
        ids = rng.permutation(num_pages)
    pt = np.full((len(seq_caps), max_pages), -1, dtype=np.int32)
    off = 0
    for b, n in enumerate(n_pages_b):
        pt[b, :n] = ids[off:off + n]
        off += int(n)
    return pt, num_pages


def poison_tail_slots(pool, page_table, seq_lens, page_size, dtype):
    """Write the NaN canary into every slot at or beyond seq_len of each request."""
    canary = {"bf16": BF16_NAN_BITS, "fp8": FP8_NAN_CODE}.get(dtype, F32_NAN_CANARY)
    for b, L in enumerate(np.asarray(seq_lens)):
        L = int(L)
        n_pages = (L + page_size - 1) // page_size
        if n_pages == 0:
            continue
        last = int(page_table[b, n_pages - 1])
        tail = L - (n_pages - 1) * page_size
        pool[last, tail:] = canary


# ----------------------------------------------------------------------------
# Decode case
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class DecodeCase:
    B: int
    H: int
    d_h: int
    r: int
    dtype: str
    page_size: int
    seq_lens: np.ndarray       # [B] int32
    page_table: np.ndarray     # [B, max_pages] int32
    num_pages: int
    q: np.ndarray              # [B, H, d_h]
    S_K: np.ndarray            # [num_pages, page_size, d_h] (or [.., G, d_h]: G groups)
    S_V: np.ndarray
    R_K: np.ndarray            # [num_pages, page_size, H, r]
    R_V: np.ndarray
    B_K: np.ndarray            # [H, d_h, r]
    B_V: np.ndarray
    scale: tuple = (1.0, 1.0, 1.0, 1.0)  # pool scales of an 8-bit ("fp8") cache

    @property
    def act_dtype(self):
        return act_dtype(self.dtype)

    @property
    def max_pages(self):
        return int(self.page_table.shape[1])

    @property
    def groups(self):
        """Shared key/value groups (1: one shared basis)."""
        return int(self.S_K.shape[2]) if self.S_K.ndim == 4 else 1

    def rows(self, b):
        """(page ids, valid tokens) of request b, in token order."""
        L = int(self.seq_lens[b])
        n = (L + self.page_size - 1) // self.page_size
        return self.page_table[b, :n], L


def make_decode_case(B, H, d_h, r, seq_lens, dtype="bf16", seed=0,
                     shuffle=False, spare_pages=0, page_size=PAGE_SIZE,
                     q_std=1.0, cache_std=1.0, base_std=None,
                     max_pages=None, fp8_scale=None, groups=1, device=None) -> DecodeCase:
    """Decode inputs: a filled paged cache plus one query row per request.

    Queries and cache rows ~ N(0, q_std^2 / cache_std^2); bases ~ N(0, 1/r)
    unless ``base_std`` is given.  With dtype "fp8" the pools hold 8-bit codes
    of value / scale (``fp8_scale``: one scale, or one per pool S_K, S_V, R_K,
    R_V; default FP8_SCALE) and the queries and bases are bf16.

    ``device`` (bf16 only; for timing runs on large workloads): the four pools
    are drawn on that torch device instead, from torch's generator seeded with
    ``seed`` (same distribution, other values, slots past a request's length
    left as drawn), and returned as bf16 torch tensors; lengths, page table,
    queries and bases are the host case's own.
    """
    rng = np.random.default_rng(seed)
    seq_lens = np.asarray(seq_lens, dtype=np.int32).reshape(B)
    pt, num_pages = make_page_table(seq_lens, page_size, shuffle, rng,
                                    spare_pages, max_pages)
    num_pages = max(num_pages, 1)
    if base_std is None:
        base_std = 1.0 / np.sqrt(r)
    adt = act_dtype(dtype)
    sc = (1.0,) * 4
    if dtype == "fp8":
        sc = fp8_scale if fp8_scale is not None else FP8_SCALE
        sc = tuple(float(x) for x in np.broadcast_to(np.asarray(sc, np.float64), (4,)))
    q = _draw(rng, (B, H, d_h), q_std, adt)
    B_K = _draw(rng, (H, d_h, r), base_std, adt)
    B_V = _draw(rng, (H, d_h, r), base_std, adt)
    # groups > 1: one shared row per group of heads, [pages, page_size, G, d_h]
    s_shape = (num_pages, page_size, d_h) if groups == 1 else (num_pages, page_size, groups, d_h)
    if device is not None:
        if dtype != "bf16":
            raise ValueError("device-drawn pools are bf16")
        pools = _device_pools(device, seed, [s_shape, s_shape, (num_pages, page_size, H, r),
                                             (num_pages, page_size, H, r)], cache_std)
        return DecodeCase(B, H, d_h, r, dtype, page_size, seq_lens, pt, num_pages,
                          q, *pools, B_K, B_V, sc)
    S_K = _draw_chunked(rng, s_shape, cache_std, dtype, scale=sc[0])
    S_V = _draw_chunked(rng, s_shape, cache_std, dtype, scale=sc[1])
    R_K = _draw_chunked(rng, (num_pages, page_size, H, r), cache_std, dtype, scale=sc[2])
    R_V = _draw_chunked(rng, (num_pages, page_size, H, r), cache_std, dtype, scale=sc[3])
    for pool in (S_K, S_V, R_K, R_V):
        poison_tail_slots(pool, pt, seq_lens, page_size, dtype)
    return DecodeCase(B, H, d_h, r, dtype, page_size, seq_lens, pt, num_pages,
                      q, S_K, S_V, R_K, R_V, B_K, B_V, sc)


def _device_pools(device, seed, shapes, std):
    """bf16 pools ~ N(0, std^2) drawn on a torch device (seeded generator, in
    chunks that bound the float32 temporary)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) + 15485863)
    out = []
    for shape in shapes:
        t = torch.empty(shape, dtype=torch.bfloat16, device=device)
        flat = t.view(-1)
        step = 1 << 26
        for a in range(0, flat.numel(), step):
            n = min(step, flat.numel() - a)
            x = torch.randn(n, generator=g, device=device, dtype=torch.float32)
            if std != 1.0:
                x.mul_(std)
            flat[a:a + n].copy_(x)
        out.append(t)
    return out


def ragged_lengths(B, lo, hi, seed):
    """Integer lengths uniform on [lo, hi] inclusive."""
    rng = np.random.default_rng(seed + 7919)
    return rng.integers(lo, hi + 1, size=B, dtype=np.int64).astype(np.int32)


# ----------------------------------------------------------------------------
# Append / prefill case
# ----------------------------------------------------------------------------
@dataclasses.dataclass
class ProjWeights:
    d: int
    H: int
    d_h: int
    r: int
    dtype: str
    W_S_K: np.ndarray   # [d_h, d]
    W_S_V: np.ndarray   # [d_h, d]
    U_K: np.ndarray     # [H, r, d]
    U_V: np.ndarray     # [H, r, d]
    B_K: np.ndarray     # [H, d_h, r]
    B_V: np.ndarray     # [H, d_h, r]
    W_Q: np.ndarray     # [H, d_h, d]  (query projection, used by harnesses only)


def make_weights(d, H, d_h, r, dtype="bf16", seed=0, groups=1) -> ProjWeights:
    """Projection weights ~ N(0, 1/d), bases ~ N(0, 1/r); W_Q drawn last.
    groups > 1: the shared weights are [groups * d_h, d] (group-major rows)."""
    rng = np.random.default_rng(seed)
    sw = 1.0 / np.sqrt(d)
    sb = 1.0 / np.sqrt(r)
    W_S_K = _draw(rng, (groups * d_h, d), sw, dtype)
    W_S_V = _draw(rng, (groups * d_h, d), sw, dtype)
    U_K = _draw(rng, (H, r, d), sw, dtype)
    U_V = _draw(rng, (H, r, d), sw, dtype)
    B_K = _draw(rng, (H, d_h, r), sb, dtype)
    B_V = _draw(rng, (H, d_h, r), sb, dtype)
    W_Q = _draw(rng, (H, d_h, d), sw, dtype)
    return ProjWeights(d, H, d_h, r, dtype, W_S_K, W_S_V, U_K, U_V, B_K, B_V, W_Q)


@dataclasses.dataclass
class AppendCase:
    X: np.ndarray           # [n, d]
    positions: np.ndarray   # [n] int32
    seq_ids: np.ndarray     # [n] int32
    page_table: np.ndarray  # [B, max_pages] int32
    num_pages: int
    page_size: int


def make_append_case(n_per_seq, start_pos, d, dtype="bf16", seed=0,
                     shuffle=True, page_size=PAGE_SIZE, x_std=None,
                     spare_pages=0, interleave=False) -> AppendCase:
    """Rows for ``len(n_per_seq)`` requests; request b appends ``n_per_seq[b]``
    rows at positions ``start_pos[b] ...``.  With ``interleave`` the rows of
    different requests are shuffled together (append must not assume order).
    """
    rng = np.random.default_rng(seed + 104729)
    n_per_seq = np.asarray(n_per_seq, dtype=np.int64)
    start_pos = np.asarray(start_pos, dtype=np.int64)
    caps = start_pos + n_per_seq
    pt, num_pages = make_page_table(caps, page_size, shuffle, rng, spare_pages)
    pos = np.concatenate([np.arange(s, s + k) for s, k in zip(start_pos, n_per_seq)]
                         ) if len(n_per_seq) else np.zeros(0, np.int64)
    sid = np.concatenate([np.full(k, b) for b, k in enumerate(n_per_seq)]
                         ) if len(n_per_seq) else np.zeros(0, np.int64)
    n = int(n_per_seq.sum())
    if interleave and n > 1:
        perm = rng.permutation(n)
        pos, sid = pos[perm], sid[perm]
    std = 1.0 / np.sqrt(d) if x_std is None else x_std
    X = _draw(rng, (n, d), std, dtype)
    return AppendCase(X, pos.astype(np.int32), sid.astype(np.int32), pt,
                      max(num_pages, 1), page_size)


def empty_pools(num_pages, page_size, H, d_h, r, dtype, canary=True, groups=1):
    """Cache pools filled with the canary (bit pattern) so untouched slots show."""
    if dtype == "bf16":
        fill = BF16_NAN_BITS if canary else np.uint16(0)
        mk = lambda shape: np.full(shape, fill, dtype=np.uint16)
    elif dtype == "fp8":
        fill = FP8_NAN_CODE if canary else np.uint8(0)
        mk = lambda shape: np.full(shape, fill, dtype=np.uint8)
    else:
        fill = F32_NAN_CANARY if canary else np.float32(0)
        mk = lambda shape: np.full(shape, fill, dtype=np.float32)
    s_shape = (num_pages, page_size, d_h) if groups == 1 else (num_pages, page_size, groups, d_h)
    return (mk(s_shape), mk(s_shape),
            mk((num_pages, page_size, H, r)), mk((num_pages, page_size, H, r)))


# ----------------------------------------------------------------------------
# The five measured workloads
# ----------------------------------------------------------------------------
CONFIGS = {
    # 1 layer, fresh 64-token prompt then one decode step, fp32 end to end.
    "tiny_fp32": dict(B=1, d=64, H=4, d_h=16, r=4, T=64, dtype="f32", seed=0),
    # decode over a 4096-token history, 16 requests, contiguous pages.
    "decode_T4096": dict(B=16, d=2048, H=16, d_h=128, r=48, T=4096, dtype="bf16", seed=0),
    # long-context decode, 4 requests x 32768 tokens.
    "decode_T32768": dict(B=4, d=4096, H=32, d_h=128, r=32, T=32768, dtype="bf16", seed=0),
    # ragged decode, 64 requests of 256..8192 tokens on shuffled 64-token pages.
    "ragged_paged": dict(B=64, H=16, d_h=128, r=56, lo=256, hi=8192, dtype="bf16", seed=0),
    # prefill + append of 8 fresh 2048-token prompts.
    "prefill_2048": dict(B=8, d=2048, H=16, d_h=128, r=48, T=2048, dtype="bf16", seed=0),
    # the 16 x 4096 decode over an 8-bit (E4M3) cache: same shapes, half the bytes
    "decode_T4096_fp8": dict(B=16, d=2048, H=16, d_h=128, r=48, T=4096, dtype="fp8", seed=0),
    # the 16 x 4096 decode with the exact rotary embedding (same cache)
    "decode_T4096_rope": dict(B=16, d=2048, H=16, d_h=128, r=48, T=4096, dtype="bf16", seed=0,
                              rope=True),
    # the 16 x 4096 decode with joint key RMSNorm (a reciprocal per head and token)
    "decode_T4096_norm": dict(B=16, d=2048, H=16, d_h=128, r=48, T=4096, dtype="bf16", seed=0,
                              norm=True),
    # the 16 x 4096 decode with a shared basis per group of 8 heads (2 groups)
    # and private rank 32: 3072 B per token against 3584 for one basis, r = 48
    "decode_T4096_g2": dict(B=16, d=2048, H=16, d_h=128, r=32, T=4096, dtype="bf16", seed=0,
                            groups=2),
}


def config_decode_case(name, seed=None, scale_T=None, device=None) -> DecodeCase:
    """Decode inputs of one of the named decode workloads (optionally with a
    shorter history ``scale_T`` for quick parity runs; ``device``: pools drawn
    on that torch device, see make_decode_case)."""
    c = CONFIGS[name]
    s = c["seed"] if seed is None else seed
    if name == "ragged_paged":
        lens = ragged_lengths(c["B"], c["lo"], c["hi"], s)
        if scale_T is not None:
            lens = np.maximum(1, (lens.astype(np.int64) * scale_T) // c["hi"]).astype(np.int32)
        return make_decode_case(c["B"], c["H"], c["d_h"], c["r"], lens, c["dtype"],
                                s, shuffle=True, spare_pages=3, device=device)
    T = c["T"] if scale_T is None else scale_T
    return make_decode_case(c["B"], c["H"], c["d_h"], c["r"], [T] * c["B"],
                            c["dtype"], s, shuffle=False, groups=c.get("groups", 1),
                            device=device)
