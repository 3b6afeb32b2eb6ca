"""PyTorch-facing binding of the LRKV C ABI.

Every function here only checks tensor properties, builds the C arguments
and calls the library on the current CUDA stream; all arithmetic runs in the
library's CUDA kernels.  Tensors must be contiguous CUDA tensors of the
cache's dtype (torch.bfloat16 or torch.float32); integer metadata is int32.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _abi

_DT = {torch.float32: _abi.LRKV_F32, torch.bfloat16: _abi.LRKV_BF16,
       torch.float8_e4m3fn: _abi.LRKV_FP8_E4M3}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, dtype=None, device=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if device and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


@dataclass
class PagedCache:
    """Caller-owned paged factored cache (four pools sharing page ids).

    S_K, S_V: [num_pages, page_size, d_h], or [num_pages, page_size, G, d_h]
    for G shared groups (head h reads group h // (H // G)); R_K, R_V:
    [num_pages, page_size, H, r].
    Pools of torch.float8_e4m3fn hold 8-bit codes whose values are the codes
    times ``scale`` (one scale per pool: S_K, S_V, R_K, R_V); the activations
    used with such a cache are bf16.  ``N_K`` ([num_pages, page_size, H] in
    the activation dtype, or None) holds the reciprocal joint key norms with
    ``norm_eps`` (see lrkv_key_norms).
    """
    S_K: torch.Tensor
    S_V: torch.Tensor
    R_K: torch.Tensor
    R_V: torch.Tensor
    scale: tuple = (1.0, 1.0, 1.0, 1.0)
    N_K: "torch.Tensor | None" = None
    norm_eps: float = 0.0

    @classmethod
    def empty(cls, num_pages, page_size, H, d_h, r, dtype=torch.bfloat16, device="cuda", groups=1):
        mk = lambda *s: torch.empty(s, dtype=dtype, device=device)
        sh = (num_pages, page_size, d_h) if groups == 1 else (num_pages, page_size, groups, d_h)
        return cls(mk(*sh), mk(*sh), mk(num_pages, page_size, H, r), mk(num_pages, page_size, H, r))

    @property
    def groups(self):
        """Shared key/value groups (1: one shared basis)."""
        return self.S_K.shape[2] if self.S_K.dim() == 4 else 1

    @property
    def dtype(self):
        return self.S_K.dtype

    @property
    def act_dtype(self):
        """dtype of every other floating tensor used with this cache."""
        return torch.bfloat16 if self.dtype == torch.float8_e4m3fn else self.dtype

    def desc(self) -> _abi.CacheDesc:
        for n in ("S_K", "S_V", "R_K", "R_V"):
            _need(getattr(self, n), n, self.dtype)
        npg, ps, d_h = self.S_K.shape[0], self.S_K.shape[1], self.S_K.shape[-1]
        _, _, H, r = self.R_K.shape
        if tuple(self.S_V.shape) != tuple(self.S_K.shape):
            raise ValueError("S_K and S_V must have the same shape")
        if self.N_K is not None:
            _need(self.N_K, "N_K", self.act_dtype)
            if tuple(self.N_K.shape) != (npg, ps, H):
                raise ValueError(f"N_K must be [{npg}, {ps}, {H}], got {tuple(self.N_K.shape)}")
        return _abi.CacheDesc(self.S_K.data_ptr(), self.S_V.data_ptr(), self.R_K.data_ptr(),
                              self.R_V.data_ptr(), npg, ps, H, d_h, r, _DT[self.dtype],
                              (ctypes.c_float * 4)(*[float(x) for x in self.scale]),
                              self.N_K.data_ptr() if self.N_K is not None else None,
                              float(self.norm_eps), self.groups)


def prefill_kernel_kind(cache: PagedCache) -> int:
    """LRKV_PREFILL_TILED or LRKV_PREFILL_PER_ROW: the attention kernel
    lrkv_prefill runs for this cache."""
    L = _abi.lib()
    st = L.lrkv_prefill_kernel_kind(ctypes.byref(cache.desc()))
    if st < 0:
        raise _abi.LrkvError("lrkv_prefill_kernel_kind", st, L)
    return st


def cache_bytes(H, d_h, r, tokens, dtype=torch.bfloat16, groups=1) -> int:
    return int(_abi.lib().lrkv_cache_bytes_grouped(H, d_h, r, groups, tokens, _DT[dtype]))


def decode_workspace_bytes(B, H, d_h, r, max_seq_len, dtype=torch.bfloat16) -> int:
    return int(_abi.lib().lrkv_decode_workspace_bytes(B, H, d_h, r, max_seq_len, _DT[dtype]))


def prefill_workspace_bytes(B, n, H, d_h, r, max_ctx, dtype=torch.bfloat16) -> int:
    return int(_abi.lib().lrkv_prefill_workspace_bytes(B, n, H, d_h, r, max_ctx, _DT[dtype]))


def workspace(nbytes, device="cuda") -> torch.Tensor:
    """A byte buffer usable as workspace (torch allocations are 256-byte aligned)."""
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def append(X, positions, seq_ids, W_S_K, W_S_V, U_K, U_V, cache: PagedCache, page_table,
           status=None, stream=None):
    """lrkv_append: project rows X and store them at (seq_ids, positions)."""
    dt = cache.act_dtype
    for n, t in (("X", X), ("W_S_K", W_S_K), ("W_S_V", W_S_V), ("U_K", U_K), ("U_V", U_V)):
        _need(t, n, dt)
    for n, t in (("positions", positions), ("seq_ids", seq_ids), ("page_table", page_table)):
        _need(t, n, torch.int32)
    if status is not None:
        _need(status, "status", torch.int32)
    n, d = X.shape
    B, max_pages = page_table.shape
    desc = cache.desc()
    code = _abi.lib().lrkv_append(_ptr(X), _ptr(positions), _ptr(seq_ids), n, d, _ptr(W_S_K),
                                  _ptr(W_S_V), _ptr(U_K), _ptr(U_V), ctypes.byref(desc),
                                  _ptr(page_table), B, max_pages, _ptr(status), _stream(stream))
    _abi.check("lrkv_append", code)


def decode(q, cache: PagedCache, B_K, B_V, seq_lens, page_table, max_seq_len, out=None,
           ws=None, status=None, stream=None):
    """lrkv_decode: per-head attention output [B, H, d_h] of one decode step."""
    dt = cache.act_dtype
    for n, t in (("q", q), ("B_K", B_K), ("B_V", B_V)):
        _need(t, n, dt)
    _need(seq_lens, "seq_lens", torch.int32)
    _need(page_table, "page_table", torch.int32)
    B, H, d_h = q.shape
    r = cache.R_K.shape[3]
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", dt)
    need = decode_workspace_bytes(B, H, d_h, r, max_seq_len, dt)
    if ws is None:
        ws = workspace(need, q.device)
    _need(ws, "ws", torch.uint8)
    desc = cache.desc()
    code = _abi.lib().lrkv_decode(_ptr(q), ctypes.byref(desc), _ptr(B_K), _ptr(B_V),
                                  _ptr(seq_lens), _ptr(page_table), B, page_table.shape[1],
                                  max_seq_len, _ptr(out), _ptr(ws), ws.numel(), _ptr(status),
                                  _stream(stream))
    _abi.check("lrkv_decode", code)
    return out


def decode_step_workspace_bytes(B, H, d_h, r, max_seq_len, dtype=torch.bfloat16) -> int:
    return _abi.lib().lrkv_decode_step_workspace_bytes(B, H, d_h, r, max_seq_len, _DT[dtype])


def decode_step(X, W_S_K, W_S_V, U_K, U_V, q, cache: PagedCache, B_K, B_V, seq_lens, page_table,
                max_seq_len, out=None, ws=None, status=None, stream=None):
    """lrkv_decode_step: append each request's new row X[b] at position
    seq_lens[b] - 1, then decode; returns out [B, H, d_h]."""
    dt = cache.act_dtype
    for n, t in (("X", X), ("W_S_K", W_S_K), ("W_S_V", W_S_V), ("U_K", U_K), ("U_V", U_V),
                 ("q", q), ("B_K", B_K), ("B_V", B_V)):
        _need(t, n, dt)
    _need(seq_lens, "seq_lens", torch.int32)
    _need(page_table, "page_table", torch.int32)
    B, H, d_h = q.shape
    r = cache.R_K.shape[3]
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", dt)
    need = decode_step_workspace_bytes(B, H, d_h, r, max_seq_len, dt)
    if ws is None:
        ws = workspace(need, q.device)
    _need(ws, "ws", torch.uint8)
    desc = cache.desc()
    code = _abi.lib().lrkv_decode_step(_ptr(X), X.shape[1], _ptr(W_S_K), _ptr(W_S_V), _ptr(U_K),
                                       _ptr(U_V), _ptr(q), ctypes.byref(desc), _ptr(B_K), _ptr(B_V),
                                       _ptr(seq_lens), _ptr(page_table), B, page_table.shape[1],
                                       max_seq_len, _ptr(out), _ptr(ws), ws.numel(), _ptr(status),
                                       _stream(stream))
    _abi.check("lrkv_decode_step", code)
    return out


def decode_step_host_workspace_bytes(B, H, d_h, r, d, max_seq_len, dtype=torch.bfloat16) -> int:
    return _abi.lib().lrkv_decode_step_host_workspace_bytes(B, H, d_h, r, d, max_seq_len, _DT[dtype])


def decode_step_host(X, W_S_K, W_S_V, U_K, U_V, q, cache: PagedCache, B_K, B_V, seq_lens,
                     page_table, max_seq_len, out=None, ws=None, status=None, stream=None):
    """lrkv_decode_step_host: the decode step with X, q, seq_lens and out in
    host memory (CPU tensors, best pinned); the copies and the step are
    enqueued on the stream, which the caller synchronises before reading out."""
    dt = cache.act_dtype
    for n, t in (("X", X), ("q", q)):
        _need(t, n, dt, device=False)
        if t.is_cuda:
            raise ValueError(f"{n} must be a host tensor")
    _need(seq_lens, "seq_lens", torch.int32, device=False)
    if seq_lens.is_cuda:
        raise ValueError("seq_lens must be a host tensor")
    for n, t in (("W_S_K", W_S_K), ("W_S_V", W_S_V), ("U_K", U_K), ("U_V", U_V), ("B_K", B_K),
                 ("B_V", B_V)):
        _need(t, n, dt)
    _need(page_table, "page_table", torch.int32)
    B, H, d_h = q.shape
    r = cache.R_K.shape[3]
    d = X.shape[1]
    if out is None:
        out = torch.empty(q.shape, dtype=dt, pin_memory=True)
    _need(out, "out", dt, device=False)
    if out.is_cuda:
        raise ValueError("out must be a host tensor")
    need = decode_step_host_workspace_bytes(B, H, d_h, r, d, max_seq_len, dt)
    if ws is None:
        ws = workspace(need, page_table.device)
    _need(ws, "ws", torch.uint8)
    desc = cache.desc()
    code = _abi.lib().lrkv_decode_step_host(_ptr(X), d, _ptr(W_S_K), _ptr(W_S_V), _ptr(U_K),
                                            _ptr(U_V), _ptr(q), ctypes.byref(desc), _ptr(B_K),
                                            _ptr(B_V), _ptr(seq_lens), _ptr(page_table), B,
                                            page_table.shape[1], max_seq_len, _ptr(out), _ptr(ws),
                                            ws.numel(), _ptr(status), _stream(stream))
    _abi.check("lrkv_decode_step_host", code)
    return out


class StepGraph:
    """lrkv_step_graph_*: the host-buffer decode step recorded once as a
    CUDA graph and replayed with one launch per step.  The graph keeps every
    tensor it was made with (held here so they stay allocated): refill X, q
    and seq_lens (pinned host tensors) between steps, launch, synchronise
    the stream, then read out."""

    def __init__(self, X, W_S_K, W_S_V, U_K, U_V, q, cache: PagedCache, B_K, B_V, seq_lens,
                 page_table, max_seq_len, out=None, ws=None, status=None):
        dt = cache.act_dtype
        for n, t in (("X", X), ("q", q)):
            _need(t, n, dt, device=False)
            if t.is_cuda or not t.is_pinned():
                raise ValueError(f"{n} must be a pinned host tensor")
        _need(seq_lens, "seq_lens", torch.int32, device=False)
        if seq_lens.is_cuda or not seq_lens.is_pinned():
            raise ValueError("seq_lens must be a pinned host tensor")
        for n, t in (("W_S_K", W_S_K), ("W_S_V", W_S_V), ("U_K", U_K), ("U_V", U_V),
                     ("B_K", B_K), ("B_V", B_V)):
            _need(t, n, dt)
        _need(page_table, "page_table", torch.int32)
        B, H, d_h = q.shape
        r, d = cache.R_K.shape[3], X.shape[1]
        if out is None:
            out = torch.empty(q.shape, dtype=dt, pin_memory=True)
        if out.is_cuda or not out.is_pinned():
            raise ValueError("out must be a pinned host tensor")
        _need(out, "out", dt, device=False)
        if ws is None:
            ws = workspace(decode_step_host_workspace_bytes(B, H, d_h, r, d, max_seq_len, dt),
                           page_table.device)
        _need(ws, "ws", torch.uint8)
        self._desc = cache.desc()
        self._keep = (X, W_S_K, W_S_V, U_K, U_V, q, cache, B_K, B_V, seq_lens, page_table, ws,
                      status)
        self.X, self.q, self.seq_lens, self.out = X, q, seq_lens, out
        h = ctypes.c_void_p()
        code = _abi.lib().lrkv_step_graph_create(
            ctypes.byref(h), _ptr(X), d, _ptr(W_S_K), _ptr(W_S_V), _ptr(U_K), _ptr(U_V), _ptr(q),
            ctypes.byref(self._desc), _ptr(B_K), _ptr(B_V), _ptr(seq_lens), _ptr(page_table), B,
            page_table.shape[1], max_seq_len, _ptr(out), _ptr(ws), ws.numel(), _ptr(status))
        _abi.check("lrkv_step_graph_create", code)
        self._h = h

    def launch(self, stream=None):
        """Enqueue one step (copies in, kernels, copy out) on the stream."""
        if self._h is None:
            raise ValueError("graph destroyed")
        _abi.check("lrkv_step_graph_launch", _abi.lib().lrkv_step_graph_launch(self._h, _stream(stream)))
        return self.out

    def close(self):
        """Destroy the graph once every launch of it has finished."""
        if self._h is not None:
            torch.cuda.synchronize()
            _abi.lib().lrkv_step_graph_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def prefill(X, Q, cu_rows, start_pos, max_ctx, W_S_K, W_S_V, U_K, U_V, B_K, B_V,
            cache: PagedCache, page_table, out=None, ws=None, status=None, stream=None):
    """lrkv_prefill: append the chunk X, then causal attention for each row's Q."""
    dt = cache.act_dtype
    for n, t in (("X", X), ("Q", Q), ("W_S_K", W_S_K), ("W_S_V", W_S_V), ("U_K", U_K),
                 ("U_V", U_V), ("B_K", B_K), ("B_V", B_V)):
        _need(t, n, dt)
    for n, t in (("cu_rows", cu_rows), ("start_pos", start_pos), ("page_table", page_table)):
        _need(t, n, torch.int32)
    n, d = X.shape
    _, H, d_h = Q.shape
    r = cache.R_K.shape[3]
    B = start_pos.shape[0]
    if out is None:
        out = torch.empty_like(Q)
    need = prefill_workspace_bytes(B, n, H, d_h, r, max_ctx, dt)
    if ws is None:
        ws = workspace(need, X.device)
    desc = cache.desc()
    code = _abi.lib().lrkv_prefill(_ptr(X), _ptr(Q), _ptr(cu_rows), _ptr(start_pos), B, n,
                                   max_ctx, d, _ptr(W_S_K), _ptr(W_S_V), _ptr(U_K), _ptr(U_V),
                                   _ptr(B_K), _ptr(B_V), ctypes.byref(desc), _ptr(page_table),
                                   page_table.shape[1], _ptr(out), _ptr(ws), ws.numel(),
                                   _ptr(status), _stream(stream))
    _abi.check("lrkv_prefill", code)
    return out


# ----------------------------------------------------------------------------
# Exact rotary position embedding (see include/lrkv.h)
# ----------------------------------------------------------------------------
class RopeTable:
    """The rotary table of lrkv_rope_table: one device buffer holding the
    (cos, sin) of position * base^(-2c/d_h) as float pairs [max_pos, d_h/2, 2]
    and, after them, the same pairs as f16."""

    def __init__(self, buf: torch.Tensor, d_h: int, max_pos: int):
        self.buf, self.d_h, self.max_pos = buf, d_h, max_pos

    @property
    def cos_sin(self) -> torch.Tensor:
        """The float pairs, [max_pos, d_h/2, 2] fp32 (a view of the buffer)."""
        n = self.max_pos * self.d_h
        return self.buf[: 4 * n].view(torch.float32).view(self.max_pos, self.d_h // 2, 2)

    @property
    def cos_sin_f16(self) -> torch.Tensor:
        """The f16 pairs, [max_pos, d_h/2, 2] (a view of the buffer)."""
        n = self.max_pos * self.d_h
        o = (4 * n + 255) // 256 * 256
        return self.buf[o: o + 2 * n].view(torch.float16).view(self.max_pos, self.d_h // 2, 2)


def rope_table_bytes(d_h, max_pos) -> int:
    return int(_abi.lib().lrkv_rope_table_bytes(d_h, max_pos))


def rope_table(d_h, max_pos, base=10000.0, device="cuda", stream=None) -> RopeTable:
    """lrkv_rope_table: (cos, sin) of position * base^(-2c/d_h) for positions
    below max_pos, in fp32 and f16."""
    nbytes = rope_table_bytes(d_h, max_pos)
    if nbytes == 0:
        raise ValueError(f"invalid rotary table size d_h={d_h} max_pos={max_pos}")
    buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
    _abi.check("lrkv_rope_table", _abi.lib().lrkv_rope_table(float(base), d_h, max_pos, _ptr(buf),
                                                             _stream(stream)))
    return RopeTable(buf, d_h, max_pos)


def decode_rope_workspace_bytes(B, H, d_h, r, max_seq_len, dtype=torch.bfloat16) -> int:
    return int(_abi.lib().lrkv_decode_rope_workspace_bytes(B, H, d_h, r, max_seq_len, _DT[dtype]))


def _need_table(table, d_h):
    if not isinstance(table, RopeTable):
        raise TypeError("table must be a RopeTable (rope_table())")
    if table.d_h != d_h:
        raise ValueError(f"table is for d_h={table.d_h}, not {d_h}")
    _need(table.buf, "table", torch.uint8)


def decode_rope(q, cache: PagedCache, B_K, B_V, seq_lens, page_table, max_seq_len, table,
                out=None, ws=None, status=None, stream=None):
    """lrkv_decode_rope: decode with the exact rotary embedding; the query of
    request b sits at position seq_lens[b] - 1."""
    dt = cache.act_dtype
    for n, t in (("q", q), ("B_K", B_K), ("B_V", B_V)):
        _need(t, n, dt)
    _need(seq_lens, "seq_lens", torch.int32)
    _need(page_table, "page_table", torch.int32)
    B, H, d_h = q.shape
    _need_table(table, d_h)
    r = cache.R_K.shape[3]
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", dt)
    if ws is None:
        ws = workspace(decode_rope_workspace_bytes(B, H, d_h, r, max_seq_len, dt), q.device)
    _need(ws, "ws", torch.uint8)
    desc = cache.desc()
    code = _abi.lib().lrkv_decode_rope(_ptr(q), ctypes.byref(desc), _ptr(B_K), _ptr(B_V),
                                       _ptr(seq_lens), _ptr(page_table), B, page_table.shape[1],
                                       max_seq_len, _ptr(table.buf), table.max_pos, _ptr(out),
                                       _ptr(ws), ws.numel(), _ptr(status), _stream(stream))
    _abi.check("lrkv_decode_rope", code)
    return out


def prefill_rope(X, Q, cu_rows, start_pos, max_ctx, W_S_K, W_S_V, U_K, U_V, B_K, B_V,
                 cache: PagedCache, page_table, table, out=None, ws=None, status=None,
                 stream=None):
    """lrkv_prefill_rope: append the chunk X, then causal attention with the
    exact rotary embedding (each row's query at its own position)."""
    dt = cache.act_dtype
    for n, t in (("X", X), ("Q", Q), ("W_S_K", W_S_K), ("W_S_V", W_S_V), ("U_K", U_K),
                 ("U_V", U_V), ("B_K", B_K), ("B_V", B_V)):
        _need(t, n, dt)
    for n, t in (("cu_rows", cu_rows), ("start_pos", start_pos), ("page_table", page_table)):
        _need(t, n, torch.int32)
    n, d = X.shape
    _, H, d_h = Q.shape
    _need_table(table, d_h)
    r = cache.R_K.shape[3]
    B = start_pos.shape[0]
    if out is None:
        out = torch.empty_like(Q)
    if ws is None:
        ws = workspace(prefill_workspace_bytes(B, n, H, d_h, r, max_ctx, dt), X.device)
    desc = cache.desc()
    code = _abi.lib().lrkv_prefill_rope(_ptr(X), _ptr(Q), _ptr(cu_rows), _ptr(start_pos), B, n,
                                        max_ctx, d, _ptr(W_S_K), _ptr(W_S_V), _ptr(U_K),
                                        _ptr(U_V), _ptr(B_K), _ptr(B_V), ctypes.byref(desc),
                                        _ptr(page_table), page_table.shape[1], _ptr(table.buf),
                                        table.max_pos, _ptr(out), _ptr(ws), ws.numel(),
                                        _ptr(status), _stream(stream))
    _abi.check("lrkv_prefill_rope", code)
    return out


def key_norms(positions, seq_ids, B_K, cache: PagedCache, page_table, status=None, stream=None):
    """lrkv_key_norms: store the reciprocal joint key norms of the given rows."""
    _need(B_K, "B_K", cache.act_dtype)
    for n, t in (("positions", positions), ("seq_ids", seq_ids), ("page_table", page_table)):
        _need(t, n, torch.int32)
    if cache.N_K is None:
        raise ValueError("cache.N_K is None")
    desc = cache.desc()
    B, max_pages = page_table.shape
    code = _abi.lib().lrkv_key_norms(_ptr(positions), _ptr(seq_ids), positions.shape[0], _ptr(B_K),
                                     ctypes.byref(desc), _ptr(page_table), B, max_pages,
                                     _ptr(status), _stream(stream))
    _abi.check("lrkv_key_norms", code)
