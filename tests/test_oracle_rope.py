"""Pins of the oracle's exact RoPE path (reading note "Low-Rank Key Value
Attention", section 8 and its figure 9), each tied to something other than
the oracle itself: the note's 2-D counterexample worked by hand, the
relative-position property of rotations, a complex-number RoPE on the
multi-query reduction, the full-rank identity basis (multi-head attention
with RoPE), the note's factored formula, and planted mistakes."""
import math

import numpy as np
import pytest

import oracle
from oracle import rope

RNG = np.random.default_rng(11)


def _case(T=7, H=3, d_h=8, r=2, seed=0):
    g = np.random.default_rng(seed)
    return (g.standard_normal((H, d_h)), g.standard_normal((T, d_h)), g.standard_normal((T, d_h)),
            g.standard_normal((T, H, r)), g.standard_normal((T, H, r)),
            g.standard_normal((H, d_h, r)) / math.sqrt(r), g.standard_normal((H, d_h, r)) / math.sqrt(r))


def test_theta_closed_form():
    np.testing.assert_allclose(rope.theta(4), [1.0, 10000.0 ** -0.5], rtol=0, atol=0)
    np.testing.assert_allclose(rope.theta(8, base=16.0), [1.0, 0.5, 0.25, 0.125], rtol=0, atol=0)


def test_rotation_by_hand():
    # (1, 0) turned by 90 degrees lands on (0, 1); (0, 1) on (-1, 0)
    np.testing.assert_allclose(rope.rotate_by([1.0, 0.0], [math.pi / 2]), [0.0, 1.0], atol=1e-15)
    np.testing.assert_allclose(rope.rotate_by([0.0, 1.0], [math.pi / 2]), [-1.0, 0.0], atol=1e-15)
    # pair (2, 3) of a 4-channel row turns by theta_1 * pos, pair (0, 1) by pos radians
    x = np.array([1.0, 0.0, 0.0, 2.0])
    y = rope.rotate(x, 3, base=16.0)   # theta = (1, 1/4)
    np.testing.assert_allclose(y, [math.cos(3), math.sin(3), -2 * math.sin(0.75), 2 * math.cos(0.75)],
                               atol=1e-15)


def test_figure_9_counterexample():
    """d_h = 2, r = 1, basis (1, 0): a key z = 1 at position 1 turns by one
    radian out of the basis' span.  A query that the rotation at position 1
    maps to the vertical axis scores sin(1) against it; any rotation of the
    one-dimensional coordinate, restored through (1, 0), stays horizontal and
    would score 0.  Worked here through the softmax by hand."""
    B = np.array([[[1.0], [0.0]]])               # [H=1, d_h=2, r=1]
    S0 = np.zeros((2, 2))                          # no shared part
    Z = np.array([[[0.0]], [[1.0]]])               # key 0 is zero, key 1 has z = 1
    V_S = np.array([[1.0, 0.0], [0.0, 1.0]])       # values: key 0 -> (1, 0), key 1 -> (0, 1)
    Z_V = np.zeros((2, 1, 1))
    q = np.array([[math.sin(1.0), math.cos(1.0)]])  # q D_1 = (0, 1)
    np.testing.assert_allclose(rope.rotate(q[0], 1), [0.0, 1.0], atol=1e-15)
    out = rope.decode_request_rope(q, 1, S0, V_S, Z, Z_V, B, B)
    s1 = math.sin(1.0) / math.sqrt(2.0)            # scores (0, sin 1) / sqrt(d_h)
    a1 = math.exp(s1) / (1.0 + math.exp(s1))
    np.testing.assert_allclose(out[0], [1 - a1, a1], rtol=1e-14)
    # the low-dimensional route: E z B^T is horizontal for every E, so both
    # scores would vanish and the weights would be equal
    assert abs(a1 - 0.5) > 0.1


def test_relative_position_shift_invariance():
    """Shifting the query and every key by the same amount changes nothing
    (D_i D_j^T = D_{i-j}); a route that depended on i + j would fail."""
    q, SK, SV, RK, RV, BK, BV = _case(seed=1)
    T = SK.shape[0]
    a = rope.decode_request_rope(q, T - 1, SK, SV, RK, RV, BK, BV, key_pos=np.arange(T))
    b = rope.decode_request_rope(q, T - 1 + 57, SK, SV, RK, RV, BK, BV, key_pos=np.arange(T) + 57)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)
    # and the rotation does matter: positions all zero give plain LRKV
    c = rope.decode_request_rope(q, 0, SK, SV, RK, RV, BK, BV, key_pos=np.zeros(T, int))
    np.testing.assert_allclose(c, oracle.decode_request(q, SK, SV, RK, RV, BK, BV), rtol=1e-12)
    assert np.abs(a - c).max() > 1e-3


def _complex_rope_mqa(q, K, V, pos_q, key_pos, base=rope.ROPE_BASE):
    """Textbook RoPE attention written with complex numbers: channel pairs
    are x_2c + i x_2c+1, multiplied by exp(i pos theta_c)."""
    d_h = K.shape[1]
    th = base ** (-np.arange(0, d_h, 2) / d_h)
    zc = lambda x: x[..., 0::2] + 1j * x[..., 1::2]
    qc = zc(q) * np.exp(1j * pos_q * th)
    kc = zc(K) * np.exp(1j * np.outer(key_pos, th))
    s = np.real(kc @ np.conj(qc)) / math.sqrt(d_h)   # Re(k conj(q)) = real dot product
    e = np.exp(s - s.max())
    return (e / e.sum()) @ V


def test_multi_query_reduction_against_complex_rope():
    """Zero private factors: every head attends the shared rows, which is
    RoPE attention with shared keys and values."""
    q, SK, SV, RK, RV, BK, BV = _case(T=9, d_h=8, seed=2)
    out = rope.decode_request_rope(q, 8, SK, SV, RK * 0, RV * 0, BK, BV)
    for h in range(q.shape[0]):
        np.testing.assert_allclose(out[h], _complex_rope_mqa(q[h], SK, SV, 8, np.arange(9)),
                                   rtol=1e-12)


def test_identity_basis_is_multi_head_rope():
    """r = d_h and B_h = I: the private coordinates are a full key, so LRKV
    with RoPE is multi-head RoPE attention on K = S + Z."""
    q, SK, SV, _, _, _, _ = _case(T=6, H=2, d_h=4, seed=3)
    g = np.random.default_rng(4)
    Z, ZV = g.standard_normal((6, 2, 4)), g.standard_normal((6, 2, 4))
    I = np.broadcast_to(np.eye(4), (2, 4, 4))
    out = rope.decode_request_rope(q, 5, SK, SV, Z, ZV, I, I)
    for h in range(2):
        np.testing.assert_allclose(out[h], _complex_rope_mqa(q[h], SK + Z[:, h], SV + ZV[:, h], 5,
                                                             np.arange(6)), rtol=1e-12)


def test_factored_formula_equals_materialised():
    for seed, (T, H, d_h, r) in enumerate([(5, 2, 4, 1), (12, 3, 8, 3), (20, 2, 16, 5)]):
        q, SK, SV, RK, RV, BK, BV = _case(T, H, d_h, r, seed=10 + seed)
        a = rope.decode_request_rope(q, T - 1, SK, SV, RK, RV, BK, BV)
        b = rope.decode_request_rope_factored(q, T - 1, SK, SV, RK, RV, BK, BV)
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)


def test_angle_addition_form_matches_materialised_scores():
    """The tensor-core decode's form of the score (q~ = q D_i; the private
    query of key j as its interleaved (cos, sin)(j theta) row C_j times the
    d_h x r matrix W with rows 2c -> q~_2c B[2c] + q~_2c+1 B[2c+1] and
    2c+1 -> q~_2c+1 B[2c] - q~_2c B[2c+1]; the shared term q~ . (S_K[j] D_j))
    equals the materialised score (q D_i) . ((S_K[j] + R_K[j] B^T) D_j)."""
    g = np.random.default_rng(21)
    for d_h, r, i in ((8, 3, 9), (16, 5, 200), (128, 48, 4095)):
        q, s, z = g.standard_normal(d_h), g.standard_normal(d_h), g.standard_normal(r)
        B = g.standard_normal((d_h, r)) / math.sqrt(r)
        qt = rope.rotate(q, i)
        W = np.empty((d_h, r))
        W[0::2] = qt[0::2, None] * B[0::2] + qt[1::2, None] * B[1::2]
        W[1::2] = qt[1::2, None] * B[0::2] - qt[0::2, None] * B[1::2]
        for j in (0, 1, i // 2, i):
            C = rope.table(d_h, j + 1)[j].reshape(-1)   # (cos, sin) interleaved by pair
            got = qt @ rope.rotate(s, j) + (C @ W) @ z
            ref = rope.rotate(q, i) @ rope.rotate(s + B @ z, j)
            assert abs(got - ref) <= 1e-12 * max(1.0, abs(ref)), (d_h, r, i, j, got, ref)


def test_paged_decode_matches_per_request():
    g = np.random.default_rng(5)
    H, d_h, r, ps = 2, 8, 2, 4
    lens = [1, 5, 9]
    pt = np.array([[3, 0, 0], [1, 4, 0], [5, 2, 6]])
    pools = [g.standard_normal((7, ps, d_h)), g.standard_normal((7, ps, d_h)),
             g.standard_normal((7, ps, H, r)), g.standard_normal((7, ps, H, r))]
    q = g.standard_normal((3, H, d_h))
    BK, BV = g.standard_normal((H, d_h, r)), g.standard_normal((H, d_h, r))
    out = rope.decode_rope(q, *pools, BK, BV, pt, lens, ps)
    for b, L in enumerate(lens):
        rows = [oracle.gather_rows(p, pt[b], L, ps) for p in pools]
        np.testing.assert_allclose(out[b], rope.decode_request_rope(q[b], L - 1, *rows, BK, BV),
                                   rtol=1e-13)


def test_table():
    t = rope.table(8, 5, base=16.0)
    assert t.shape == (5, 4, 2)
    np.testing.assert_allclose(t[3, 2], [math.cos(3 * 0.25), math.sin(3 * 0.25)], rtol=1e-15)


@pytest.mark.parametrize("mutation", ["half_split", "sign", "query_only", "absolute_sum"])
def test_mutations_fail(monkeypatch, mutation):
    """A plausible mistake in the rotation fails one of the pins above."""
    orig = rope.rotate_by

    def bad(x, angles):
        x = np.asarray(x, np.float64)
        a = np.asarray(angles, np.float64)
        if mutation == "half_split":   # pairs (c, c + d_h/2) instead of (2c, 2c+1)
            n = x.shape[-1] // 2
            y = np.concatenate([x[..., :n] * np.cos(a) - x[..., n:] * np.sin(a),
                                x[..., :n] * np.sin(a) + x[..., n:] * np.cos(a)], axis=-1)
            return y
        if mutation == "sign":
            return orig(x, -a)
        return orig(x, a)

    monkeypatch.setattr(rope, "rotate_by", bad)
    failed = False
    checks = [test_rotation_by_hand, test_figure_9_counterexample, test_multi_query_reduction_against_complex_rope,
              test_identity_basis_is_multi_head_rope, test_relative_position_shift_invariance]
    if mutation == "query_only":      # keys left unrotated
        monkeypatch.setattr(rope, "rotate", lambda x, pos, base=rope.ROPE_BASE:
                            orig(np.asarray(x, np.float64), np.asarray(pos, np.float64)[..., None]
                                 * rope.theta(np.asarray(x).shape[-1], base)) if np.ndim(pos) == 0
                            else np.asarray(x, np.float64))
    if mutation == "absolute_sum":    # query turned the wrong way: scores depend on i + j
        monkeypatch.setattr(rope, "rotate", lambda x, pos, base=rope.ROPE_BASE:
                            orig(np.asarray(x, np.float64), (-1 if np.ndim(pos) == 0 else 1)
                                 * np.asarray(pos, np.float64)[..., None]
                                 * rope.theta(np.asarray(x).shape[-1], base)))
    for chk in checks:
        try:
            chk()
        except AssertionError:
            failed = True
    assert failed, mutation
