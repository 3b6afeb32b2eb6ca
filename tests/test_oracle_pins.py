"""Pins of the float64 oracle against what the LRKV reading note and plain
mathematics fix: the printed worked example, closed-form budgets, brute force
on tiny inputs, special cases that reduce to textbook attention, and
invariants.  Mutation tests at the end plant plausible mistakes in the oracle
(on the CPU) and check that a pin catches each one.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
from scipy.special import softmax

import lrkv_inputs as I
import oracle
from oracle import lrkv_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------
# Independent brute force (explicit loops; exp without max subtraction)
# ----------------------------------------------------------------------------
def brute_decode_one(q, sk, sv, rk, rv, bk, bv):
    """One head, one query: loops over every scalar; no library matmul."""
    T, d_h = len(sk), len(sk[0])
    r = len(rk[0])
    keys, vals = [], []
    for j in range(T):
        kj, vj = [], []
        for c in range(d_h):
            ak, av = sk[j][c], sv[j][c]
            for k in range(r):
                ak += rk[j][k] * bk[c][k]
                av += rv[j][k] * bv[c][k]
            kj.append(ak)
            vj.append(av)
        keys.append(kj)
        vals.append(vj)
    w = []
    for j in range(T):
        s = 0.0
        for c in range(d_h):
            s += q[c] * keys[j][c]
        w.append(math.exp(s / math.sqrt(d_h)))
    Z = sum(w)
    return [sum(w[j] * vals[j][c] for j in range(T)) / Z for c in range(d_h)]


def check_bruteforce(seed=0):
    rng = np.random.default_rng(seed)
    for trial in range(6):
        d_h = int(rng.integers(2, 17))
        r = int(rng.integers(1, 4))
        H = int(rng.integers(1, 4))
        Bn = int(rng.integers(1, 3))
        lens = rng.integers(1, 9, size=Bn)
        case = I.make_decode_case(Bn, H, d_h, r, lens, dtype="f32",
                                  seed=seed * 31 + trial, shuffle=True,
                                  spare_pages=2, page_size=4)
        f = lambda a: I.to_f64(a, "f32")
        got = O.decode(f(case.q), f(case.S_K), f(case.S_V), f(case.R_K), f(case.R_V),
                       f(case.B_K), f(case.B_V), case.page_table, case.seq_lens, 4)
        for b in range(Bn):
            L = int(lens[b])
            pages = case.page_table[b]
            rows = lambda pool: [pool[pages[t // 4], t % 4] for t in range(L)]
            sk, sv = rows(f(case.S_K)), rows(f(case.S_V))
            rk, rv = rows(f(case.R_K)), rows(f(case.R_V))
            for h in range(H):
                want = brute_decode_one(
                    list(f(case.q)[b, h]), [list(x) for x in sk], [list(x) for x in sv],
                    [list(x[h]) for x in rk], [list(x[h]) for x in rv],
                    [list(x) for x in f(case.B_K)[h]], [list(x) for x in f(case.B_V)[h]])
                assert np.allclose(got[b, h], want, rtol=1e-12, atol=1e-13), (trial, b, h)


def check_worked_example():
    g = _load("worked_example.json")
    q = np.array(g["q"], float)
    S = np.array([g["shared_key"]], float)
    R = np.array([g["private_key_coordinate"]], float)
    Bk = np.array(g["expansion_column_B_K"], float)
    K = O.expand_head(S, R, Bk)
    assert np.array_equal(K[0], g["materialised_key"])
    assert float(q @ K[0]) == g["score_materialised"]
    # Scores seen through the oracle's softmax: a second key of zeros gives a
    # weight ratio exp(9 / sqrt(2)) under the 1/sqrt(d_h) scale.
    d_h = 2
    Sk = np.vstack([S, np.zeros((1, 2))])
    Rk = np.vstack([R, np.zeros((1, 1))])
    V = np.eye(2)
    for fn in (O.decode_request, O.decode_request_factored):
        w = fn(q[None], Sk, V, Rk[:, None, :], np.zeros((2, 1, 1)),
               Bk[None], np.zeros((1, 2, 1)))[0]
        want = g["score_factored"] / math.sqrt(d_h)
        assert math.isclose(math.log(w[0] / w[1]), want, rel_tol=1e-12)
    # Value side: weights 1/4 and 3/4 over private coordinates 2 and 6,
    # expansion column (1, -1) -> (5, -5).  Keys chosen so the softmax gives
    # exactly those weights: score gap ln 3.
    gap = math.log(3.0) * math.sqrt(d_h)
    Sk = np.array([[0.0, 0.0], [gap, 0.0]])
    Rv = np.array(g["private_value_coordinates"], float)[:, None, :]
    Bv = np.array(g["expansion_column_B_V"], float)[None]
    for fn in (O.decode_request, O.decode_request_factored):
        o = fn(np.array([[1.0, 0.0]]), Sk, np.zeros((2, 2)), np.zeros((2, 1, 1)), Rv,
               np.zeros((1, 2, 1)), Bv)[0]
        assert np.allclose(o, g["expanded_value"], rtol=0, atol=1e-12)


def check_mqa_reduction(seed=3):
    """Zero private factors: every head attends to the shared S_K/S_V alone,
    i.e. multi-query attention (section 3: small random init starts near
    multi-query; page on MHA/MQA/GQA)."""
    rng = np.random.default_rng(seed)
    T, H, d_h, r = 37, 3, 8, 2
    sk, sv = rng.standard_normal((T, d_h)), rng.standard_normal((T, d_h))
    rk, rv = rng.standard_normal((T, H, r)), rng.standard_normal((T, H, r))
    q = rng.standard_normal((H, d_h))
    z = np.zeros((H, d_h, r))
    o = O.decode_request(q, sk, sv, rk, rv, z, z)
    for h in range(H):
        a = softmax(sk @ q[h] / np.sqrt(d_h))
        assert np.allclose(o[h], a @ sv, rtol=1e-12, atol=1e-14)


# ----------------------------------------------------------------------------
# Pins
# ----------------------------------------------------------------------------
def test_worked_example():
    check_worked_example()


def test_bruteforce_tiny_paged():
    check_bruteforce()


def test_mqa_reduction():
    check_mqa_reduction()


def test_single_row_is_expanded_value():
    rng = np.random.default_rng(1)
    H, d_h, r = 4, 16, 4
    q = rng.standard_normal((H, d_h))
    sk, sv = rng.standard_normal((1, d_h)), rng.standard_normal((1, d_h))
    rk, rv = rng.standard_normal((1, H, r)), rng.standard_normal((1, H, r))
    bk, bv = rng.standard_normal((H, d_h, r)), rng.standard_normal((H, d_h, r))
    o = O.decode_request(q, sk, sv, rk, rv, bk, bv)
    for h in range(H):
        assert np.allclose(o[h], sv[0] + bv[h] @ rv[0, h], rtol=1e-14, atol=1e-14)


def test_zero_query_gives_mean_value():
    rng = np.random.default_rng(2)
    T, H, d_h, r = 11, 2, 6, 3
    sk, sv = rng.standard_normal((T, d_h)), rng.standard_normal((T, d_h))
    rk, rv = rng.standard_normal((T, H, r)), rng.standard_normal((T, H, r))
    bk, bv = rng.standard_normal((H, d_h, r)), rng.standard_normal((H, d_h, r))
    o = O.decode_request(np.zeros((H, d_h)), sk, sv, rk, rv, bk, bv)
    for h in range(H):
        V = sv + rv[:, h, :] @ bv[h].T
        assert np.allclose(o[h], V.mean(axis=0), rtol=1e-13, atol=1e-14)


def test_factored_equals_materialised():
    rng = np.random.default_rng(4)
    T, H, d_h, r = 300, 5, 32, 7
    args = (rng.standard_normal((H, d_h)) * 2, rng.standard_normal((T, d_h)),
            rng.standard_normal((T, d_h)), rng.standard_normal((T, H, r)),
            rng.standard_normal((T, H, r)), rng.standard_normal((H, d_h, r)),
            rng.standard_normal((H, d_h, r)))
    a = O.decode_request(*args)
    b = O.decode_request_factored(*args)
    assert np.max(np.abs(a - b)) <= 1e-12 * np.max(np.abs(a))


def test_near_cancelling_shared_and_private():
    """Shared key and private correction nearly cancel (section 9 asks for
    this case): the materialised key is tiny, and brute force still agrees."""
    d_h, r = 4, 1
    sk = np.array([[1.0, -2.0, 0.5, 3.0], [0.3, 0.1, -0.2, 0.4]])
    bk = np.array([[1.0], [-2.0], [0.5], [3.0]])[None]
    rk = np.array([[[-1.0 + 1e-9]], [[0.0]]])
    sv = np.array([[1.0, 0, 0, 0], [0, 1.0, 0, 0]])
    rv = np.zeros((2, 1, 1))
    bv = np.zeros((1, d_h, 1))
    q = np.array([[5.0, 1.0, -3.0, 2.0]])
    o = O.decode_request(q, sk, sv, rk, rv, bk, bv)[0]
    want = brute_decode_one(list(q[0]), sk.tolist(), sv.tolist(), rk[:, 0].tolist(),
                            rv[:, 0].tolist(), bk[0].tolist(), bv[0].tolist())
    assert np.allclose(o, want, rtol=1e-12, atol=1e-15)
    K0 = O.expand_head(sk, rk[:, 0], bk[0])[0]
    assert np.max(np.abs(K0)) < 1e-8


def test_branches_must_merge_before_softmax():
    """Section 2: scores (2,0) and (0,2) from the two branches.  Merged they
    give equal weights; normalised separately and each reading its own value
    they give something else.  The oracle follows the merged form."""
    s_shared, s_private = np.array([2.0, 0.0]), np.array([0.0, 2.0])
    merged = softmax(s_shared + s_private)
    assert np.allclose(merged, [0.5, 0.5])
    v_shared, v_private = np.array([1.0, 0.0]), np.array([0.0, 1.0])
    sep = softmax(s_shared) @ v_shared + softmax(s_private) @ v_private
    both = merged @ (v_shared + v_private)
    assert not np.isclose(sep, both)
    # The oracle with d_h = 1: keys 2 and 0 shared, 0 and 2 private (r = 1,
    # B = 1), q = sqrt(1) so the scale is 1.
    o = O.decode_request(np.array([[1.0]]), np.array([[2.0], [0.0]]),
                         np.array([[1.0], [0.0]]), np.array([[[0.0]], [[2.0]]]),
                         np.array([[[0.0]], [[1.0]]]), np.ones((1, 1, 1)),
                         np.ones((1, 1, 1)))
    assert np.isclose(o[0, 0], both)


def test_scale_is_head_width_not_rank():
    """Section 2 / Algorithm 2: divide by sqrt(d_h).  With 1/sqrt(r) the
    weights of the worked example would change."""
    q = np.array([2.0, 1.0])
    K = np.array([[5.0, -1.0], [0.0, 0.0]])
    o = O.attend(q, K, np.eye(2))
    assert math.isclose(math.log(o[0] / o[1]), 9 / math.sqrt(2), rel_tol=1e-12)
    assert not math.isclose(math.log(o[0] / o[1]), 9 / math.sqrt(1), rel_tol=1e-6)


def test_causal_mask_hides_later_rows():
    rng = np.random.default_rng(5)
    K, V = rng.standard_normal((6, 4)), rng.standard_normal((6, 4))
    q = rng.standard_normal(4)
    vis = np.arange(6) <= 2
    a = softmax(K[:3] @ q / 2.0)
    assert np.allclose(O.attend(q, K, V, vis), a @ V[:3], rtol=1e-13)


def test_placement_golden():
    g = _load("placement_small.json")
    ps = g["page_size"]
    pt = np.array(g["page_table"], np.int32)
    rows = g["rows"]
    n = len(rows)
    H, d_h, r = 2, 3, 2
    pools = I.empty_pools(5, ps, H, d_h, r, "f32", canary=True)
    pools = [p.astype(np.float64) for p in pools]
    vals = [np.arange(n * d_h, dtype=float).reshape(n, d_h) + 1,
            -np.arange(n * d_h, dtype=float).reshape(n, d_h) - 1,
            np.arange(n * H * r, dtype=float).reshape(n, H, r) + 100,
            -np.arange(n * H * r, dtype=float).reshape(n, H, r) - 100]
    pos = np.array([x["position"] for x in rows])
    sid = np.array([x["seq_id"] for x in rows])
    out = O.place(pools, vals, pos, sid, pt, ps)
    touched = np.zeros((5, ps), bool)
    for i, x in enumerate(rows):
        pg, sl = x["page"], x["slot"]
        touched[pg, sl] = True
        for k in range(4):
            assert np.array_equal(out[k][pg, sl], vals[k][i])
    for k in range(4):
        assert np.all(np.isnan(out[k][~touched]))


def test_place_gather_round_trip_shuffled():
    ac = I.make_append_case([13, 70, 1], [0, 5, 63], d=8, dtype="f32", seed=3,
                            shuffle=True, spare_pages=2, interleave=True)
    n = len(ac.positions)
    vals = [np.random.default_rng(k).standard_normal((n, 3)) for k in range(2)] + \
           [np.random.default_rng(k).standard_normal((n, 2, 2)) for k in range(2, 4)]
    pools = [p.astype(np.float64) for p in I.empty_pools(ac.num_pages, 64, 2, 3, 2, "f32")]
    out = O.place(pools, vals, ac.positions, ac.seq_ids, ac.page_table, 64)
    for b in range(3):
        idx = np.where(ac.seq_ids == b)[0]
        idx = idx[np.argsort(ac.positions[idx])]
        p0 = int(ac.positions[idx[0]])
        got = O.gather_rows(out[0], ac.page_table[b], p0 + len(idx), 64)[p0:]
        assert np.array_equal(got, vals[0][idx])


def test_projection_matches_effective_weight():
    """X W_h = S + R_h B_h^T with W_h = W_S + U_h B_h^T (section 3, eqs 2-5),
    written in the paper's orientation from the stored output-major weights.
    Non-square shapes so a transposed operand cannot pass."""
    w = I.make_weights(d=12, H=3, d_h=5, r=2, dtype="f32", seed=9)
    f = lambda a: I.to_f64(a, "f32")
    X = np.random.default_rng(0).standard_normal((7, 12))
    S_K, S_V, R_K, R_V = O.project(X, f(w.W_S_K), f(w.W_S_V), f(w.U_K), f(w.U_V))
    for h in range(3):
        W_eff = f(w.W_S_K).T + f(w.U_K)[h].T @ f(w.B_K)[h].T    # d x d_h
        assert np.allclose(X @ W_eff, O.expand_head(S_K, R_K[:, h], f(w.B_K)[h]),
                           rtol=1e-12, atol=1e-12)
    # one-hot rows pick single input columns of each weight
    E = np.eye(12)[[3, 0, 11]]
    S_K, _, R_K, _ = O.project(E, f(w.W_S_K), f(w.W_S_V), f(w.U_K), f(w.U_V))
    assert np.array_equal(S_K[0], f(w.W_S_K)[:, 3])
    assert np.array_equal(R_K[2, 1], f(w.U_K)[1, :, 11])


def test_prefill_equals_row_by_row_decode():
    """Prefill's causal attention over a fresh chunk equals a decode of each
    row over the rows up to and including itself."""
    w = I.make_weights(d=16, H=2, d_h=8, r=3, dtype="f32", seed=4)
    f = lambda a: I.to_f64(a, "f32")
    ac = I.make_append_case([9, 5], [0, 0], d=16, dtype="f32", seed=2,
                            shuffle=True, interleave=True)
    n = len(ac.positions)
    Q = np.random.default_rng(7).standard_normal((n, 2, 8))
    X = f(ac.X)
    out = O.prefill(Q, X, ac.positions, ac.seq_ids, f(w.W_S_K), f(w.W_S_V), f(w.U_K),
                    f(w.U_V), f(w.B_K), f(w.B_V))
    rows = O.project(X, f(w.W_S_K), f(w.W_S_V), f(w.U_K), f(w.U_V))
    pools = [p.astype(np.float64) for p in I.empty_pools(ac.num_pages, 64, 2, 8, 3, "f32")]
    pools = O.place(pools, rows, ac.positions, ac.seq_ids, ac.page_table, 64)
    for i in range(n):
        b, p = int(ac.seq_ids[i]), int(ac.positions[i])
        one = O.decode(Q[i][None], *pools, f(w.B_K), f(w.B_V), ac.page_table[b:b + 1],
                       np.array([p + 1]), 64)
        assert np.allclose(out[i], one[0], rtol=1e-12, atol=1e-14)


def test_prefill_bruteforce_tiny():
    w = I.make_weights(d=6, H=2, d_h=3, r=2, dtype="f32", seed=11)
    f = lambda a: I.to_f64(a, "f32")
    X = np.random.default_rng(3).standard_normal((4, 6))
    Q = np.random.default_rng(4).standard_normal((4, 2, 3))
    pos, sid = np.arange(4), np.zeros(4, int)
    out = O.prefill(Q, X, pos, sid, f(w.W_S_K), f(w.W_S_V), f(w.U_K), f(w.U_V),
                    f(w.B_K), f(w.B_V))
    Wk, Wv, Uk, Uv = f(w.W_S_K), f(w.W_S_V), f(w.U_K), f(w.U_V)
    for i in range(4):
        for h in range(2):
            sk = [[sum(X[j][t] * Wk[c][t] for t in range(6)) for c in range(3)] for j in range(i + 1)]
            sv = [[sum(X[j][t] * Wv[c][t] for t in range(6)) for c in range(3)] for j in range(i + 1)]
            rk = [[sum(X[j][t] * Uk[h][k][t] for t in range(6)) for k in range(2)] for j in range(i + 1)]
            rv = [[sum(X[j][t] * Uv[h][k][t] for t in range(6)) for k in range(2)] for j in range(i + 1)]
            want = brute_decode_one(list(Q[i, h]), sk, sv, rk, rv, f(w.B_K)[h].tolist(),
                                    f(w.B_V)[h].tolist())
            assert np.allclose(out[i, h], want, rtol=1e-11, atol=1e-13)


# ----------------------------------------------------------------------------
# Budgets (section 4, equation 9 and the printed values)
# ----------------------------------------------------------------------------
def test_budget_numbers():
    g = _load("budgets.json")
    for e in g["payload_ratio"]:
        pct = float(O.payload_ratio(e["H"], e["d_h"], e["r"])) * 100
        assert round(pct, e["digits"]) == e["percent"], e
    t = g["table12_bytes"]
    assert round(t["lrkv"] / t["mha"] * 100, 2) == t["percent"]
    assert round(float(O.payload_ratio(18, 128, 64)) * 100, 2) == t["percent"]
    for e in g["max_rank"]:
        assert O.max_rank(e["d_h"], e["H"], Fraction(e["c_num"], e["c_den"])) == e["r_max"]
    MiB = 1 << 20
    for e in g["payload_mib"]:
        assert O.mha_payload(e["bytes_per_elem"], e["N"], e["B"], e["T"], e["H"], e["d_h"]) / MiB == e["mha_mib"]
        assert O.lrkv_payload(e["bytes_per_elem"], e["N"], e["B"], e["T"], e["H"], e["d_h"], e["r"]) / MiB == e["lrkv_mib"]
    p = g["param_ratio"]
    assert round(float(O.param_ratio(p["H"], p["d_h"], p["r"], p["d"])) * 100, 1) == p["percent"]
    a = g["decode_arith_ratio_long_context"]
    assert round(float(O.decode_arith_ratio(a["d_h"], a["r"], 10 ** 9)), 2) == a["limit"]
    rp = g["replicated"]
    assert round(float(O.replicated_ratio(1, rp["H"], rp["r"], rp["d_h"])) * 100, 1) == rp["single_percent"]
    assert round(float(O.replicated_ratio(rp["P"], rp["H"], rp["r"], rp["d_h"])) * 100, 1) == rp["replicated_percent"]


def test_config_ratios():
    """Payload ratios of the measured decode shapes through equation 9."""
    assert O.payload_ratio(16, 128, 48) == Fraction(7, 16)       # 0.4375
    assert O.payload_ratio(32, 128, 32) == Fraction(9, 32)       # 0.28125
    assert O.payload_ratio(16, 128, 56) == Fraction(1, 2)
    assert O.payload_ratio(4, 16, 4) == Fraction(1, 2)


def test_decode_byte_model_closed_form():
    # per visible token: keys and values, d_h shared + H r private, 2 bytes
    lens = [4096] * 16
    assert O.decode_bytes(lens, 16, 128, 48) == (
        65536 * (2 * 128 + 2 * 16 * 48) * 2 + 2 * 16 * 128 * 48 * 2 + 2 * 16 * 16 * 128 * 2)
    assert O.decode_bytes(lens, 16, 128, 48) == 235_405_312


# ----------------------------------------------------------------------------
# Mutation tests: each plants one plausible mistake in the oracle and checks
# that some pin above catches it.
# ----------------------------------------------------------------------------
def _must_fail(check):
    with pytest.raises(AssertionError):
        check()


def test_mutation_dropped_private_term(monkeypatch):
    monkeypatch.setattr(O, "expand_head", lambda S, R, B: np.asarray(S, float))
    _must_fail(check_bruteforce)
    _must_fail(check_worked_example)


def test_mutation_sign_of_private_term(monkeypatch):
    real = O.expand_head
    monkeypatch.setattr(O, "expand_head", lambda S, R, B: 2 * np.asarray(S, float) - real(S, R, B))
    _must_fail(check_bruteforce)


def test_mutation_scale_by_rank(monkeypatch):
    real = O.attend

    def wrong(q, K, V, visible=None):  # scale 1/sqrt(d_h/2) instead of 1/sqrt(d_h)
        return real(np.asarray(q) * math.sqrt(2.0), K, V, visible)
    monkeypatch.setattr(O, "attend", wrong)
    _must_fail(check_bruteforce)
    _must_fail(check_worked_example)


def test_mutation_off_by_one_visibility(monkeypatch):
    real = O.gather_rows
    monkeypatch.setattr(O, "gather_rows", lambda pool, pages, n, ps: real(pool, pages, max(n - 1, 1), ps))
    _must_fail(check_bruteforce)


def test_mutation_head_index(monkeypatch):
    real = O.expand_head

    def wrong_decode_request(q, S_K, S_V, R_K, R_V, B_K, B_V):
        H = q.shape[0]
        out = np.empty((H, S_K.shape[1]))
        for h in range(H):
            hh = (h + 1) % H
            out[h] = O.attend(q[h], real(S_K, R_K[:, hh], B_K[h]), real(S_V, R_V[:, h], B_V[h]))
        return out
    monkeypatch.setattr(O, "decode_request", wrong_decode_request)

    def check():
        rng = np.random.default_rng(0)
        T, H, d_h, r = 9, 3, 4, 2
        args = [rng.standard_normal(s) for s in
                [(H, d_h), (T, d_h), (T, d_h), (T, H, r), (T, H, r), (H, d_h, r), (H, d_h, r)]]
        assert np.allclose(O.decode_request(*args), O.decode_request_factored(*args))
    _must_fail(check)


def test_mutation_transposed_base(monkeypatch):
    real = O.expand_head
    monkeypatch.setattr(O, "expand_head",
                        lambda S, R, B: np.asarray(S, float) + (np.asarray(R) @ np.asarray(B).T[::-1, ::-1]))
    _must_fail(check_bruteforce)


def test_decode_flop_model_matches_arithmetic_ratio():
    """The flop model divided by the dense-MHA flops of the same step is the
    section 4 decode arithmetic ratio 1 + r/d_h + r/T (one request)."""
    for T, H, d_h, r in [(4096, 16, 128, 48), (32768, 32, 128, 32), (7, 3, 16, 4)]:
        dense = 2 * (T * H * 2 * d_h)
        assert Fraction(O.decode_flops([T], H, d_h, r), dense) == O.decode_arith_ratio(d_h, r, T)
