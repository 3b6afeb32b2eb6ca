"""Exact rotary position embedding (RoPE) over the factored cache, float64.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module.

Source: the reading note "Low-Rank Key Value Attention | 共享缓存与逐头残差",
section 8 ("can RoPE's rotation pass through the low-rank basis").  The
note shows (figure 9, a 2-D example with a rank-1 basis) that rotating the
r-dimensional private coordinate cannot stand in for rotating the expanded
private key: that needs E_j B_h^T = B_h^T D_j, which fails whenever the
rotation carries the key out of the basis' span.  Its exact alternative
keeps the private coordinates z_j unrotated and scores each key at its own
position:  q~_i (z_j B_h^T D_j)^T = (q~_i D_j^T B_h) z_j^T.  The rotation is
linear, so it distributes over the shared and private terms of the key
(section 8, first step), and the full key of head h at position j is
(s_j + z_j B_h^T) D_j, the query at position i is q~_i = q_i D_i.  Values
are not rotated.

Readings (the note fixes no convention):
  * D_j is the rotation of the original rotary embedding: channel pairs
    (2c, 2c+1) of a row vector x turn by angle j * theta_c,
        (x_2c, x_2c+1) -> (x_2c cos - x_2c+1 sin, x_2c sin + x_2c+1 cos),
    theta_c = base^(-2c / d_h), base 10000, over all d_h channels;
  * key j of a request sits at position j (0-based), the decode query at
    position seq_len - 1; a prefill row's query at its own position;
  * the cache keeps S_K, S_V, R_K, R_V unrotated (the linear projections of
    Algorithm 1), so append is unchanged and the rotation is applied where
    scores are formed.

The materialised path below is the plain definition (expand each head's
keys, rotate keys and query, textbook attention).  The factored path is the
note's formula, used only to cross-check the oracle.
"""
from __future__ import annotations

import math

import numpy as np

from .lrkv_oracle import attend, expand_head, gather_rows

ROPE_BASE = 10000.0


def theta(d_h, base=ROPE_BASE):
    """Angle per position of channel pair c: base^(-2c/d_h), c < d_h/2."""
    c = np.arange(d_h // 2, dtype=np.float64)
    return base ** (-2.0 * c / d_h)


def rotate_by(x, angles):
    """Turn channel pairs (2c, 2c+1) of row vectors x [..., d_h] by angles
    [..., d_h/2] (the rotation D of the section-8 formulas)."""
    x = np.asarray(x, np.float64)
    a = np.asarray(angles, np.float64)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    c, s = np.cos(a), np.sin(a)
    out = np.empty(np.broadcast_shapes(x.shape[:-1], a.shape[:-1]) + (x.shape[-1],), np.float64)
    out[..., 0::2] = x0 * c - x1 * s
    out[..., 1::2] = x0 * s + x1 * c
    return out


def rotate(x, pos, base=ROPE_BASE):
    """x D_pos: rows x [..., d_h] at integer positions pos [...] (broadcast)."""
    x = np.asarray(x, np.float64)
    pos = np.asarray(pos, np.float64)
    return rotate_by(x, pos[..., None] * theta(x.shape[-1], base))


def decode_request_rope(q, pos_q, S_K, S_V, R_K, R_V, B_K, B_V, key_pos=None, base=ROPE_BASE):
    """Per-head output of one query at position pos_q over T cached rows.

    q: [H, d_h] (unrotated); S_K, S_V: [T, d_h]; R_K, R_V: [T, H, r];
    B_K, B_V: [H, d_h, r]; key_pos: [T] positions of the rows (default
    0..T-1).  All rows are visible.  Materialise K_h = S_K + R_K[h] B_K[h]^T,
    rotate each key by its position and the query by pos_q, attend over the
    unrotated V_h = S_V + R_V[h] B_V[h]^T.
    """
    q = np.asarray(q, np.float64)
    H, d_h = q.shape
    T = S_K.shape[0]
    kp = np.arange(T) if key_pos is None else np.asarray(key_pos)
    out = np.empty((H, d_h), np.float64)
    for h in range(H):
        K_h = rotate(expand_head(S_K, R_K[:, h, :], B_K[h]), kp, base)
        V_h = expand_head(S_V, R_V[:, h, :], B_V[h])
        out[h] = attend(rotate(q[h], pos_q, base), K_h, V_h)
    return out


def decode_request_rope_factored(q, pos_q, S_K, S_V, R_K, R_V, B_K, B_V, key_pos=None,
                                 base=ROPE_BASE):
    """The same through the note's exact formula: the shared key cached
    rotated, s_j D_j, and the private score (q~ D_j^T B_h) z_j^T formed per
    key position; values as in equation 7.  Cross-check only."""
    q = np.asarray(q, np.float64)
    H, d_h = q.shape
    T = S_K.shape[0]
    kp = np.arange(T) if key_pos is None else np.asarray(key_pos)
    s_rot = rotate(S_K, kp, base)                      # cached s_j D_j
    out = np.empty((H, d_h), np.float64)
    for h in range(H):
        qt = rotate(q[h], pos_q, base)                 # q~_i
        s = np.empty(T)
        for j in range(T):
            u = rotate(qt, -kp[j], base)               # q~_i D_j^T (D_j^T = D_{-j})
            s[j] = qt @ s_rot[j] + (u @ B_K[h]) @ R_K[j, h, :]
        s /= math.sqrt(d_h)
        e = np.exp(s - s.max())
        a = e / e.sum()
        out[h] = a @ S_V + (a @ R_V[:, h, :]) @ B_V[h].T
    return out


def decode_rope(q, S_K, S_V, R_K, R_V, B_K, B_V, page_table, seq_lens, page_size, pairs=None,
                base=ROPE_BASE):
    """Batched decode from paged pools with RoPE: request b's query sits at
    position seq_lens[b] - 1 and its key j at position j.  Returns
    out [B, H, d_h] (NaN where ``pairs`` leaves a (b, h) out)."""
    Bn, H, d_h = q.shape
    out = np.full((Bn, H, d_h), np.nan)
    want = None
    if pairs is not None:
        want = {}
        for b, h in pairs:
            want.setdefault(int(b), []).append(int(h))
    for b in range(Bn):
        if want is not None and b not in want:
            continue
        L = int(seq_lens[b])
        pages = page_table[b]
        rows = [gather_rows(p, pages, L, page_size) for p in (S_K, S_V, R_K, R_V)]
        heads = range(H) if want is None else want[b]
        for h in heads:
            K_h = rotate(expand_head(rows[0], rows[2][:, h, :], B_K[h]), np.arange(L), base)
            V_h = expand_head(rows[1], rows[3][:, h, :], B_V[h])
            out[b, h] = attend(rotate(q[b, h], L - 1, base), K_h, V_h)
    return out


def table(d_h, max_pos, base=ROPE_BASE):
    """cos and sin of delta * theta_c for delta < max_pos: [max_pos, d_h/2, 2]."""
    a = np.arange(max_pos, dtype=np.float64)[:, None] * theta(d_h, base)[None, :]
    return np.stack([np.cos(a), np.sin(a)], axis=-1)
