"""Plain float64 oracle of Low-Rank Key Value attention (LRKV).

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module.

Source: the reading note "Low-Rank Key Value Attention | 共享缓存与逐头残差"
(Zhongzhu Zhou, on O'Neill, Clancy, Matskevichus and Reid, arXiv 2601.11471).
Citations below name that note's sections, equations and algorithms.

What LRKV computes.  Each layer keeps one shared key projection W_S_K and one
shared value projection W_S_V (width d_h), and each head h a low-rank pair
U_h (d x r), B_h (d_h x r).  The head's effective projection is
W_h = W_S + U_h B_h^T, so X W_h = S + R_h B_h^T with S = X W_S (shared,
cached once per token) and R_h = X U_h (private, r wide, cached per head)
(section 3, the chain of equations 2-5).  Decode from that cache is
*exactly* ordinary softmax attention over the materialised keys and values
K_h = S_K + R_K[h] B_K[h]^T, V_h = S_V + R_V[h] B_V[h]^T (section 3,
Algorithm 2: "mathematically the same as expanding first"), so the oracle
is that plain definition: expand, then textbook attention with scale
1/sqrt(d_h) and a causal mask (section 2, the three-line definition of
s, a and o; the scale is the original head width, not sqrt(r)).

A second, factored path (section 3, equations 6 and 7) exists only so the
tests can check the oracle against itself; it never feeds a comparison with
the CUDA path.

Readings where the note is silent:
  * the current decode token is visible to itself (causal j <= i): decode
    runs after the new row has been appended (Algorithm 1 tracks sequence
    boundaries for the causal mask, section 2 says decode adds one new row);
  * the query projection and the output projection / head concatenation
    (first and last steps of Algorithm 2) stay outside: q is an input and the
    output is the per-head o_h;
  * no RoPE and no RMSNorm (Algorithm 1 is "the linear projection version").

Parity pins for every function live in tests/test_oracle_pins.py.
"""
from __future__ import annotations

from fractions import Fraction
import math
import numpy as np

__all__ = [
    "expand_head", "attend", "decode_request", "decode_request_factored",
    "gather_rows", "decode", "project", "place", "prefill",
    "payload_ratio", "max_rank", "mha_payload", "lrkv_payload",
    "param_ratio", "decode_arith_ratio", "replicated_ratio",
    "decode_bytes", "decode_flops",
]


# ----------------------------------------------------------------------------
# Attention (section 2; section 3 equations 2-5; Algorithm 2)
# ----------------------------------------------------------------------------
def expand_head(S, R_h, B_h):
    """K_h = S + R_h B_h^T (section 3, equations 2-5).

    S: [T, d_h], R_h: [T, r], B_h: [d_h, r]  ->  [T, d_h]
    """
    S = np.asarray(S, dtype=np.float64)
    return S + np.asarray(R_h, np.float64) @ np.asarray(B_h, np.float64).T


def attend(q, K, V, visible=None):
    """Textbook single-query softmax attention (section 2).

    s_j = q . K_j / sqrt(d_h) + m_j,  a = softmax(s),  o = sum_j a_j V_j,
    with m_j = 0 on visible rows and -inf elsewhere.  d_h is the key width.
    q: [d_h], K, V: [T, d_h], visible: optional [T] bool.
    """
    q = np.asarray(q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    d_h = K.shape[1]
    s = (K @ q) / math.sqrt(d_h)
    if visible is not None:
        s = np.where(np.asarray(visible, bool), s, -np.inf)
    m = np.max(s)
    e = np.exp(s - m)
    a = e / e.sum()
    return a @ V


def decode_request(q, S_K, S_V, R_K, R_V, B_K, B_V):
    """Per-head decode output for one request, by materialising K_h and V_h.

    q: [H, d_h]; S_K, S_V: [T, d_h] (all T rows visible); R_K, R_V: [T, H, r];
    B_K, B_V: [H, d_h, r].  Returns o: [H, d_h] (before head concatenation
    and the output projection).
    """
    H = q.shape[0]
    out = np.empty((H, S_K.shape[1]), np.float64)
    for h in range(H):
        K_h = expand_head(S_K, R_K[:, h, :], B_K[h])
        V_h = expand_head(S_V, R_V[:, h, :], B_V[h])
        out[h] = attend(q[h], K_h, V_h)
    return out


def decode_request_factored(q, S_K, S_V, R_K, R_V, B_K, B_V):
    """Same result through the reassociated forms (section 3, eqs 6 and 7).

    Scores: q_h S_K^T + (q_h B_K[h]) R_K[h]^T, with the private query
    p = q_h B_K[h] formed once.  Values: a_h S_V + (a_h R_V[h]) B_V[h]^T, the
    private reduction expanded once.  Used only to cross-check the oracle.
    """
    H, d_h = q.shape
    out = np.empty((H, d_h), np.float64)
    for h in range(H):
        p = q[h] @ B_K[h]
        s = (S_K @ q[h] + R_K[:, h, :] @ p) / math.sqrt(d_h)
        e = np.exp(s - s.max())
        a = e / e.sum()
        out[h] = a @ S_V + (a @ R_V[:, h, :]) @ B_V[h].T
    return out


# ----------------------------------------------------------------------------
# Paged cache access (section 3: shared and private pages share one token
# numbering and one lifetime)
# ----------------------------------------------------------------------------
def gather_rows(pool, pages, n_tokens, page_size):
    """Rows 0..n_tokens-1 of one request, read page by page in token order."""
    pool = np.asarray(pool)
    rows = []
    for t in range(n_tokens):
        rows.append(pool[int(pages[t // page_size]), t % page_size])
    if not rows:
        return np.zeros((0,) + pool.shape[2:], pool.dtype)
    return np.stack(rows)


def decode(q, S_K, S_V, R_K, R_V, B_K, B_V, page_table, seq_lens, page_size,
           pairs=None):
    """Decode for a batch read from paged pools (all arguments float64).

    Returns out [B, H, d_h]; with ``pairs`` (list of (b, h)) only those heads
    are computed and the rest are NaN.
    """
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
        sk = gather_rows(S_K, pages, L, page_size)
        sv = gather_rows(S_V, pages, L, page_size)
        rk = gather_rows(R_K, pages, L, page_size)
        rv = gather_rows(R_V, pages, L, page_size)
        heads = range(H) if want is None else want[b]
        for h in heads:
            K_h = expand_head(sk, rk[:, h, :], B_K[h])
            V_h = expand_head(sv, rv[:, h, :], B_V[h])
            out[b, h] = attend(q[b, h], K_h, V_h)
    return out


# ----------------------------------------------------------------------------
# Cache build / append (section 3, Algorithm 1)
# ----------------------------------------------------------------------------
def project(X, W_S_K, W_S_V, U_K, U_V):
    """Shared and private projections of new rows (Algorithm 1; eqs 2-5).

    Weights are stored output-major: W_S_*: [d_h, d], U_*: [H, r, d], so
    S_K = X W_S_K^T (the paper's X W_S) and R_K[h] = X U_K[h]^T (X U_h).
    Returns S_K, S_V: [n, d_h] and R_K, R_V: [n, H, r].
    """
    X = np.asarray(X, np.float64)
    S_K = X @ np.asarray(W_S_K, np.float64).T
    S_V = X @ np.asarray(W_S_V, np.float64).T
    R_K = np.einsum("nd,hrd->nhr", X, np.asarray(U_K, np.float64))
    R_V = np.einsum("nd,hrd->nhr", X, np.asarray(U_V, np.float64))
    return S_K, S_V, R_K, R_V


def place(pools, rows, positions, seq_ids, page_table, page_size):
    """Write each row's four blocks at its token position (Algorithm 1).

    Row i of request seq_ids[i] at position positions[i] goes to page
    page_table[seq_ids[i], positions[i] // page_size], slot
    positions[i] % page_size, in all four pools under the same page id.
    Returns copies of the pools; untouched slots keep their contents.
    """
    out = [np.array(p, copy=True) for p in pools]
    for i in range(len(positions)):
        b, pos = int(seq_ids[i]), int(positions[i])
        page = int(page_table[b, pos // page_size])
        slot = pos % page_size
        for k in range(4):
            out[k][page, slot] = rows[k][i]
    return out


def prefill(Q, X, positions, seq_ids, W_S_K, W_S_V, U_K, U_V, B_K, B_V,
            history=None, rows_wanted=None, heads_wanted=None):
    """Causal LRKV attention of a chunk of new rows (section 2 prefill).

    Each new row i (request seq_ids[i], position positions[i], query
    Q[i]: [H, d_h]) attends to every row of its request at positions
    <= positions[i]: earlier history (``history[b]`` = (S_K, S_V, R_K, R_V)
    float64 rows 0..P-1) followed by the chunk's own projected rows.
    Returns out [n, H, d_h] (NaN for rows/heads not wanted).
    """
    Q = np.asarray(Q, np.float64)
    n, H, d_h = Q.shape
    S_K, S_V, R_K, R_V = project(X, W_S_K, W_S_V, U_K, U_V)
    out = np.full((n, H, d_h), np.nan)
    rows_wanted = range(n) if rows_wanted is None else rows_wanted
    heads_wanted = range(H) if heads_wanted is None else heads_wanted
    by_req = {}
    for i in range(n):
        by_req.setdefault(int(seq_ids[i]), []).append(i)
    full = {}
    for b, idx in by_req.items():
        P = 0 if history is None or b not in history else history[b][0].shape[0]
        T = P + len(idx)
        sk = np.zeros((T, d_h)); sv = np.zeros((T, d_h))
        rk = np.zeros((T, H, R_K.shape[2])); rv = np.zeros_like(rk)
        filled = np.zeros(T, bool)
        if P:
            hk, hv, hrk, hrv = history[b]
            sk[:P], sv[:P], rk[:P], rv[:P] = hk, hv, hrk, hrv
            filled[:P] = True
        for i in idx:
            p = int(positions[i])
            sk[p], sv[p], rk[p], rv[p] = S_K[i], S_V[i], R_K[i], R_V[i]
            filled[p] = True
        full[b] = (sk, sv, rk, rv, filled)
    for i in rows_wanted:
        b, p = int(seq_ids[i]), int(positions[i])
        sk, sv, rk, rv, filled = full[b]
        assert filled[: p + 1].all(), "a visible row was never written"
        visible = np.arange(sk.shape[0]) <= p
        for h in heads_wanted:
            K_h = expand_head(sk, rk[:, h, :], B_K[h])
            V_h = expand_head(sv, rv[:, h, :], B_V[h])
            out[i, h] = attend(Q[i, h], K_h, V_h, visible)
    return out


# ----------------------------------------------------------------------------
# Budgets and cost models (section 4)
# ----------------------------------------------------------------------------
def mha_payload(b, N, B, T, H, d_h):
    """M_MHA = 2 b N B T H d_h bytes (section 2, the cache payload formula)."""
    return 2 * b * N * B * T * H * d_h


def lrkv_payload(b, N, B, T, H, d_h, r):
    """M_LRKV = 2 b N B T (d_h + H r) bytes (section 4, equation 9)."""
    return 2 * b * N * B * T * (d_h + H * r)


def payload_ratio(H, d_h, r):
    """M_LRKV / M_MHA = 1/H + r/d_h as an exact fraction (section 4, eq 9)."""
    return Fraction(1, H) + Fraction(r, d_h)


def max_rank(d_h, H, c):
    """Largest rank within a cache budget c: floor(d_h (c - 1/H)) (eq 9).

    ``c`` may be a Fraction for exact arithmetic.
    """
    c = Fraction(c) if not isinstance(c, Fraction) else c
    return math.floor(d_h * (c - Fraction(1, H)))


def param_ratio(H, d_h, r, d):
    """K/V projection parameters, LRKV over MHA: 1/H + (r/d_h)(1 + d_h/d)
    (section 4, parameter cost)."""
    return Fraction(1, H) + Fraction(r, d_h) * (1 + Fraction(d_h, d))


def decode_arith_ratio(d_h, r, T):
    """(2 T d_h + 2 T r + 2 r d_h) / (2 T d_h) = 1 + r/d_h + r/T (section 4)."""
    return Fraction(2 * T * d_h + 2 * T * r + 2 * r * d_h, 2 * T * d_h)


def replicated_ratio(P, H, r, d_h):
    """Payload ratio when heads are split over P devices that each keep the
    shared block: P/H + r/d_h (section 4, tensor parallelism)."""
    return Fraction(P, H) + Fraction(r, d_h)


def decode_bytes(seq_lens, H, d_h, r, elem_bytes=2):
    """Algorithmic bytes of one decode step: every visible cache row once
    (shared d_h + per-head r, keys and values), both bases, q and out."""
    T = int(np.sum(np.asarray(seq_lens, dtype=np.int64)))
    Bn = len(seq_lens)
    cache = T * 2 * (d_h + H * r) * elem_bytes
    bases = 2 * H * d_h * r * elem_bytes
    qo = 2 * Bn * H * d_h * elem_bytes
    return cache + bases + qo


def decode_flops(seq_lens, H, d_h, r):
    """Multiply-add count x2 of one decode step through the factored cache:
    per visible row and head, d_h + r for the score and d_h + r for the
    value; per head 2 r d_h for the private query and the expansion."""
    T = int(np.sum(np.asarray(seq_lens, dtype=np.int64)))
    Bn = len(seq_lens)
    return 2 * (T * H * 2 * (d_h + r) + Bn * H * 2 * r * d_h)
