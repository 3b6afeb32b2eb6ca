"""Joint RMSNorm of the keys over the factored cache, float64.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module.

Source: the reading note "Low-Rank Key Value Attention | 共享缓存与逐头残差",
section 8 ("RMSNorm still has a per-head joint quantity").  A normalised key
divides the full key k_{h,j} = s_j + z_j B_h^T by its root mean square
n_{h,j}, and expanding the square gives
    d_h n_{h,j}^2 = |s_j|^2 + 2 s_j B_h z_j^T + z_j B_h^T B_h z_j^T + d_h eps,
a cross term that ties the shared and private parts together: normalising
the two paths separately turns the key.  The note's exact scheme (without
RoPE) computes 1 / n_{h,j} when the token is appended, stores it per head
and position, and multiplies it onto the sum of the two score terms; a fixed
per-channel gain moves to the query side.

Readings where the note leaves a choice open:
  * the library applies only 1 / n_{h,j}; a per-channel gain g is folded
    into the query by the caller (q g . k / n = q . (k g) / n), as is the
    query's own normalisation;
  * eps is a model constant given with the cache;
  * the norm is that of the cached key (the oracle's float64 projection,
    the kernels' stored values).

The plain definition is ``decode_request_norm``: materialise every head's
keys, divide each by its root mean square, textbook attention.  The factored
route (the note's expansion and the stored reciprocal) is a cross-check.
"""
from __future__ import annotations

import math

import numpy as np

from .lrkv_oracle import attend, expand_head, gather_rows


def rms_normalise(K, eps):
    """Rows of K divided by their root mean square sqrt(mean(k^2) + eps)."""
    K = np.asarray(K, np.float64)
    return K / np.sqrt(np.mean(K * K, axis=-1, keepdims=True) + eps)


def inv_norm(S, R_h, B_h, eps):
    """1 / n_{h,j} of every row: the reciprocal root mean square of the full
    key s_j + z_j B_h^T.  S: [T, d_h], R_h: [T, r], B_h: [d_h, r] -> [T]."""
    K = expand_head(S, R_h, B_h)
    return 1.0 / np.sqrt(np.mean(K * K, axis=-1) + eps)


def inv_norm_expanded(S, R_h, B_h, eps):
    """The same through the note's expansion of d_h n^2 (cross-check)."""
    S = np.asarray(S, np.float64)
    Z = np.asarray(R_h, np.float64)
    B = np.asarray(B_h, np.float64)
    d_h = S.shape[1]
    sq = (np.sum(S * S, axis=1) + 2.0 * np.einsum("td,dr,tr->t", S, B, Z)
          + np.einsum("tr,dr,de,te->t", Z, B, B, Z) + d_h * eps)
    return 1.0 / np.sqrt(sq / d_h)


def key_norms(S_K, R_K, B_K, eps):
    """Stored reciprocals for rows [T]: S_K [T, d_h], R_K [T, H, r],
    B_K [H, d_h, r] -> [T, H]."""
    H = B_K.shape[0]
    return np.stack([inv_norm(S_K, R_K[:, h, :], B_K[h], eps) for h in range(H)], axis=1)


def decode_request_norm(q, S_K, S_V, R_K, R_V, B_K, B_V, eps):
    """Per-head output with RMS-normalised keys (plain definition).
    q: [H, d_h] (gain and query normalisation already applied)."""
    q = np.asarray(q, np.float64)
    H, d_h = q.shape
    out = np.empty((H, d_h), np.float64)
    for h in range(H):
        K_h = rms_normalise(expand_head(S_K, R_K[:, h, :], B_K[h]), eps)
        V_h = expand_head(S_V, R_V[:, h, :], B_V[h])
        out[h] = attend(q[h], K_h, V_h)
    return out


def decode_request_norm_factored(q, S_K, S_V, R_K, R_V, B_K, B_V, eps):
    """The note's exact scheme: (q.s_j + (q B_h).z_j) / n_{h,j} with 1/n from
    the expanded square, then equation 7 for the values (cross-check)."""
    q = np.asarray(q, np.float64)
    H, d_h = q.shape
    out = np.empty((H, d_h), np.float64)
    for h in range(H):
        p = q[h] @ B_K[h]
        w = inv_norm_expanded(S_K, R_K[:, h, :], B_K[h], eps)
        s = (S_K @ q[h] + R_K[:, h, :] @ p) * w / math.sqrt(d_h)
        e = np.exp(s - s.max())
        a = e / e.sum()
        out[h] = a @ S_V + (a @ R_V[:, h, :]) @ B_V[h].T
    return out


def decode_norm(q, S_K, S_V, R_K, R_V, B_K, B_V, N_K, page_table, seq_lens, page_size,
                pairs=None):
    """Batched decode from paged pools, scores multiplied by the stored
    reciprocal norms N_K [pages, page_size, H] (whatever they hold: the
    parity tests pass the values the kernels stored).  Returns [B, H, d_h]."""
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
        sk, sv, rk, rv, nk = (gather_rows(p, pages, L, page_size) for p in (S_K, S_V, R_K, R_V, N_K))
        for h in (range(H) if want is None else want[b]):
            K_h = expand_head(sk, rk[:, h, :], B_K[h]) * nk[:, h][:, None]
            V_h = expand_head(sv, rv[:, h, :], B_V[h])
            out[b, h] = attend(q[b, h], K_h, V_h)
    return out
