"""Times the float64 oracle on host cores (test infrastructure only).

Used by bench.py's CPU-baseline leg and its ``--impl reference`` arm.  The
oracle runs as it stands: for each sampled (request, head) pair it gathers the
request's rows from the paged pools, materialises K_h and V_h and runs
textbook softmax attention.  Work is spread over a ``spawn`` process pool of
single-threaded workers (BLAS threads pinned to 1), so ``cores`` is exactly
the number of worker processes.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import time

_CASE = None


_ROPE = False
_NORM = False


def _init(config):
    global _CASE, _ROPE, _NORM
    import lrkv_inputs as I
    _CASE = I.config_decode_case(config)
    _ROPE = bool(I.CONFIGS[config].get("rope"))
    _NORM = bool(I.CONFIGS[config].get("norm"))


def _run_pairs(pairs):
    import numpy as np
    import lrkv_inputs as I
    from . import lrkv_oracle as O
    from . import fp8, grouped, norm, rope
    c = _CASE
    f = lambda a: I.to_f64(a, c.act_dtype)
    if c.dtype == "fp8":  # 8-bit pools: codes times the pool's scale
        fp = lambda a, k: fp8.dequantize(a, c.scale[k])
    else:
        fp = lambda a, k: I.to_f64(a, c.dtype)
    t0 = time.perf_counter()
    for b, h in pairs:
        pages, L = c.rows(b)
        sk = fp(O.gather_rows(c.S_K, pages, L, c.page_size), 0)
        sv = fp(O.gather_rows(c.S_V, pages, L, c.page_size), 1)
        if c.groups > 1:  # pools [pages, page_size, G, d_h]: this head's group
            g = grouped.group_of(h, c.H, c.groups)
            sk, sv = sk[:, g, :], sv[:, g, :]
        rk = fp(O.gather_rows(c.R_K, pages, L, c.page_size)[:, h, :], 2)
        rv = fp(O.gather_rows(c.R_V, pages, L, c.page_size)[:, h, :], 3)
        K_h = O.expand_head(sk, rk, f(c.B_K[h]))
        V_h = O.expand_head(sv, rv, f(c.B_V[h]))
        qh = f(c.q[b, h])
        if _NORM:  # joint key RMSNorm (eps 1e-6)
            K_h = norm.rms_normalise(K_h, 1e-6)
        if _ROPE:  # keys at positions 0..L-1, the query at L-1
            K_h, qh = rope.rotate(K_h, np.arange(L)), rope.rotate(qh, L - 1)
        o = O.attend(qh, K_h, V_h)
        assert np.all(np.isfinite(o))
    return time.perf_counter() - t0


def time_oracle_decode(config: str, n_pairs: int, workers: int | None = None, seed: int = 0):
    """Run the oracle on ``n_pairs`` sampled (request, head) pairs of a decode
    workload; returns dict(wall_s, cpu_s, pairs, cores, heads)."""
    import numpy as np
    import lrkv_inputs as I
    cfg = I.CONFIGS[config]
    B, H = cfg["B"], cfg["H"]
    workers = max(1, min(workers or os.cpu_count() or 1, n_pairs))
    rng = np.random.default_rng(seed)
    pairs = [(int(rng.integers(B)), int(rng.integers(H))) for _ in range(n_pairs)]
    chunks = [pairs[i::workers] for i in range(workers)]
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS",
                                             "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"
    try:
        ctx = mp.get_context("spawn")
        with ctx.Pool(workers, initializer=_init, initargs=(config,)) as pool:
            pool.map(_run_pairs, [[(0, 0)]] * workers)   # warm: imports, page-in
            t0 = time.perf_counter()
            cpu = pool.map(_run_pairs, chunks)
            wall = time.perf_counter() - t0
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    return dict(wall_s=wall, cpu_s=float(sum(cpu)), pairs=n_pairs, cores=workers, heads=H)


_PF = None


def _init_prefill(config):
    """The prefill workload's inputs, drawn as bench.py draws them: rows of
    request b are X[b T : (b + 1) T] at positions 0 .. T - 1."""
    global _PF
    import numpy as np
    import lrkv_inputs as I
    c = I.CONFIGS[config]
    B, d, H, d_h, r, T = c["B"], c["d"], c["H"], c["d_h"], c["r"], c["T"]
    ac = I.make_append_case([T] * B, [0] * B, d, dtype="bf16", seed=c["seed"], shuffle=True)
    w = I.make_weights(d, H, d_h, r, "bf16", seed=c["seed"])
    rng = np.random.default_rng(99)
    Q = I.f32_to_bf16_bits(rng.standard_normal((B * T, H, d_h)).astype(np.float32))
    _PF = (c, ac.X, Q, w)


def _run_prefill_request(job):
    """Request b of the prefill workload through the oracle: the projection
    of its T rows (timed alone), then oracle.prefill for k sampled rows and
    all heads (which projects again); returns (t_proj, t_attn, k, T)."""
    import numpy as np
    import lrkv_inputs as I
    from . import lrkv_oracle as O
    b, k, seed = job
    c, X, Q, w = _PF
    T = c["T"]
    f = lambda a: I.to_f64(a, "bf16")
    Xb, Qb = f(X[b * T:(b + 1) * T]), f(Q[b * T:(b + 1) * T])
    Ws = [f(w.W_S_K), f(w.W_S_V), f(w.U_K), f(w.U_V)]
    Bk, Bv = f(w.B_K), f(w.B_V)
    rows = np.random.default_rng(seed).choice(T, size=k, replace=False)
    t0 = time.perf_counter()
    O.project(Xb, *Ws)
    t1 = time.perf_counter()
    out = O.prefill(Qb, Xb, np.arange(T), np.full(T, b), *Ws, Bk, Bv, rows_wanted=rows)
    t2 = time.perf_counter()
    assert np.all(np.isfinite(out[rows]))
    return t1 - t0, max(0.0, (t2 - t1) - (t1 - t0)), k, T


def time_oracle_prefill(config: str, k_rows: int, workers: int | None = None):
    """The oracle's prefill of the fresh-prompt workload on host cores: each
    process takes one request (b = process index), times the projection of
    its T rows and the causal attention of k_rows sampled rows (all heads),
    and scales to a full request: T / (t_proj + t_attn T / k).  Processes run
    concurrently, so the job's tokens/s is the sum of theirs.  Returns
    dict(tokens_per_s, wall_s, cpu_s, cores, rows_sampled)."""
    import lrkv_inputs as I
    B = I.CONFIGS[config]["B"]
    workers = max(1, min(workers or os.cpu_count() or 1, B))
    saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS",
                                             "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"
    try:
        ctx = mp.get_context("spawn")
        with ctx.Pool(workers, initializer=_init_prefill, initargs=(config,)) as pool:
            t0 = time.perf_counter()
            res = pool.map(_run_prefill_request, [(b, k_rows, 100 + b) for b in range(workers)])
            wall = time.perf_counter() - t0
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    rate = sum(T / (tp + ta * T / k) for tp, ta, k, T in res)
    return dict(tokens_per_s=rate, wall_s=wall, cpu_s=float(sum(tp * 2 + ta for tp, ta, _, _ in res)),
                cores=workers, rows_sampled=k_rows * workers)
