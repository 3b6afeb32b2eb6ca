"""Grouped shared basis: one shared key/value projection per group of heads,
float64.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module.

Source: the reading note "Low-Rank Key Value Attention | 共享缓存与逐头残差",
section 3, after equations 2-5: one shared basis saves the most memory, but
when the heads fall naturally into groups with very different needs, each
group may get a basis of its own; the price is storing several copies of
the shared features, the gain depends on how far the private rank can then
drop.  With G groups, head h of group g(h) has the effective projection
W_h = W_S^{g(h)} + U_h B_h^T, so a token caches G shared rows S^g = X W_S^g
(width d_h each) and the per-head private rows R_h = X U_h, and
    K_h = S_K^{g(h)} + R_K[h] B_K[h]^T,   V_h = S_V^{g(h)} + R_V[h] B_V[h]^T.
G = 1 is the single shared basis of the rest of the note; G = H with no
private part is multi-head attention, and 1 < G < H with no private part is
grouped-query attention.

Readings where the note leaves a choice open:
  * groups are runs of consecutive heads of equal size: g(h) = h // (H / G),
    G divides H;
  * a token's shared row holds the G groups one after another
    ([G, d_h], group-major), and the shared weights are stored the same way
    ([G d_h, d], output-major, like the single-basis W_S);
  * the cache payload per token and layer is 2 (G d_h + H r) elements, so
    the ratio to multi-head attention (2 H d_h) is G/H + r/d_h (section 4,
    equation 9 with G shared rows).
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

from .lrkv_oracle import attend, expand_head, gather_rows


def group_of(h, H, G):
    """The group of head h: consecutive runs of H / G heads."""
    if H % G:
        raise ValueError("G must divide H")
    return h // (H // G)


def project_grouped(X, W_S_K, W_S_V, U_K, U_V, G):
    """Shared rows of the G groups and private rows of new tokens.

    W_S_*: [G d_h, d] (group-major, output-major rows); U_*: [H, r, d].
    Returns S_K, S_V: [n, G, d_h] and R_K, R_V: [n, H, r].
    """
    X = np.asarray(X, np.float64)
    n = X.shape[0]
    S_K = (X @ np.asarray(W_S_K, np.float64).T).reshape(n, G, -1)
    S_V = (X @ np.asarray(W_S_V, np.float64).T).reshape(n, G, -1)
    R_K = np.einsum("nd,hrd->nhr", X, np.asarray(U_K, np.float64))
    R_V = np.einsum("nd,hrd->nhr", X, np.asarray(U_V, np.float64))
    return S_K, S_V, R_K, R_V


def decode_request_grouped(q, S_K, S_V, R_K, R_V, B_K, B_V):
    """Per-head output of one query over T rows (all visible), materialising
    each head's keys and values from its group's shared rows.

    q: [H, d_h]; S_K, S_V: [T, G, d_h]; R_K, R_V: [T, H, r]; B: [H, d_h, r].
    """
    q = np.asarray(q, np.float64)
    H, d_h = q.shape
    G = S_K.shape[1]
    out = np.empty((H, d_h), np.float64)
    for h in range(H):
        g = group_of(h, H, G)
        K_h = expand_head(S_K[:, g, :], R_K[:, h, :], B_K[h])
        V_h = expand_head(S_V[:, g, :], R_V[:, h, :], B_V[h])
        out[h] = attend(q[h], K_h, V_h)
    return out


def decode_grouped(q, S_K, S_V, R_K, R_V, B_K, B_V, page_table, seq_lens, page_size,
                   pairs=None):
    """Batched decode from paged pools (S pools [pages, page_size, G, d_h]).
    Returns out [B, H, d_h] (NaN where ``pairs`` leaves a (b, h) out)."""
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
        rows = [gather_rows(p, page_table[b], L, page_size) for p in (S_K, S_V, R_K, R_V)]
        G = rows[0].shape[1]
        for h in (range(H) if want is None else want[b]):
            g = group_of(h, H, G)
            K_h = expand_head(rows[0][:, g, :], rows[2][:, h, :], B_K[h])
            V_h = expand_head(rows[1][:, g, :], rows[3][:, h, :], B_V[h])
            out[b, h] = attend(q[b, h], K_h, V_h)
    return out


def payload_ratio_grouped(H, d_h, r, G):
    """Cache payload against multi-head attention: (G d_h + H r) / (H d_h)."""
    return Fraction(G * d_h + H * r, H * d_h)
