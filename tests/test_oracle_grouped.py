"""Pins of the oracle's grouped shared basis (reading note "Low-Rank Key
Value Attention", section 3 after equations 2-5: a basis per group of heads),
each tied to something other than the function under test: values worked by
hand, the single-basis oracle (G = 1), multi-head and grouped-query
attention written out with a plain softmax (no private part), the byte
model's closed form, and planted mistakes."""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import grouped


def _softmax_attend(q, K, V):
    s = K @ q / math.sqrt(K.shape[1])
    w = np.exp(s - s.max())
    return (w / w.sum()) @ V


def _case(T, H, G, d_h, r, seed):
    g = np.random.default_rng(seed)
    return (g.standard_normal((H, d_h)), g.standard_normal((T, G, d_h)), g.standard_normal((T, G, d_h)),
            g.standard_normal((T, H, r)), g.standard_normal((T, H, r)),
            g.standard_normal((H, d_h, r)) / math.sqrt(r), g.standard_normal((H, d_h, r)) / math.sqrt(r))


def test_group_of():
    assert [grouped.group_of(h, 8, 2) for h in range(8)] == [0, 0, 0, 0, 1, 1, 1, 1]
    assert [grouped.group_of(h, 6, 3) for h in range(6)] == [0, 0, 1, 1, 2, 2]
    with pytest.raises(ValueError):
        grouped.group_of(0, 6, 4)


def test_single_row_by_hand():
    """One row: every softmax weight is 1, so o_h = S_V^{g(h)} + R_V[h] B_V[h]^T
    exactly.  H = 2 heads in G = 2 groups, d_h = 2, r = 1."""
    q = np.array([[1.0, 0.0], [0.0, 1.0]])
    S_K = np.zeros((1, 2, 2))
    S_V = np.array([[[1.0, 2.0], [3.0, 4.0]]])
    R_K = np.zeros((1, 2, 1))
    R_V = np.array([[[1.0], [2.0]]])
    B = np.array([[[1.0], [0.0]], [[0.0], [1.0]]])
    out = grouped.decode_request_grouped(q, S_K, S_V, R_K, R_V, B, B)
    np.testing.assert_array_equal(out, [[2.0, 2.0], [3.0, 6.0]])


def test_zero_query_averages_by_hand():
    """q = 0 gives uniform weights: o_h is the mean of its group's value rows
    plus the mean private expansion.  H = 4, G = 2 (heads 0-1 and 2-3)."""
    q = np.zeros((4, 2))
    S_K = np.ones((2, 2, 2))
    S_V = np.array([[[0.0, 4.0], [8.0, 0.0]], [[2.0, 0.0], [0.0, 6.0]]])
    R = np.zeros((2, 4, 1))
    B = np.zeros((4, 2, 1))
    out = grouped.decode_request_grouped(q, S_K, S_V, R, R, B, B)
    np.testing.assert_array_equal(out, [[1.0, 2.0], [1.0, 2.0], [4.0, 3.0], [4.0, 3.0]])


def test_one_group_is_the_single_basis_oracle():
    q, SK, SV, RK, RV, BK, BV = _case(9, 4, 1, 8, 3, seed=1)
    a = grouped.decode_request_grouped(q, SK, SV, RK, RV, BK, BV)
    b = oracle.decode_request(q, SK[:, 0], SV[:, 0], RK, RV, BK, BV)
    np.testing.assert_allclose(a, b, rtol=1e-14, atol=1e-14)


def test_no_private_part_is_multi_head_and_grouped_query_attention():
    """With B = 0 the private rows drop out: G = H is multi-head attention
    (each head its own keys and values), 1 < G < H grouped-query attention
    (the heads of a group share them)."""
    for H, G in ((4, 4), (4, 2), (6, 3)):
        q, SK, SV, RK, RV, BK, BV = _case(7, H, G, 8, 2, seed=H + G)
        BK[:] = 0
        BV[:] = 0
        out = grouped.decode_request_grouped(q, SK, SV, RK, RV, BK, BV)
        for h in range(H):
            g = h // (H // G)
            np.testing.assert_allclose(out[h], _softmax_attend(q[h], SK[:, g], SV[:, g]), rtol=1e-13)


def test_heads_of_a_group_share_the_shared_rows():
    """Changing group 1's shared rows leaves the heads of group 0 untouched."""
    q, SK, SV, RK, RV, BK, BV = _case(5, 4, 2, 8, 2, seed=3)
    a = grouped.decode_request_grouped(q, SK, SV, RK, RV, BK, BV)
    SK2, SV2 = SK.copy(), SV.copy()
    SK2[:, 1] += 1.0
    SV2[:, 1] -= 2.0
    b = grouped.decode_request_grouped(q, SK2, SV2, RK, RV, BK, BV)
    np.testing.assert_array_equal(a[:2], b[:2])
    assert np.all(np.abs(a[2:] - b[2:]) > 1e-6)


def test_projection_by_hand_and_against_single_basis():
    X = np.array([[1.0, 2.0]])
    W = np.array([[1.0, 0.0], [0.0, 1.0], [1.0, 1.0], [2.0, -1.0]])  # G = 2 groups of d_h = 2
    U = np.zeros((1, 1, 2))
    SK, SV, RK, RV = grouped.project_grouped(X, W, 2 * W, U, U, 2)
    np.testing.assert_array_equal(SK, [[[1.0, 2.0], [3.0, 0.0]]])
    np.testing.assert_array_equal(SV, [[[2.0, 4.0], [6.0, 0.0]]])
    g = np.random.default_rng(4)
    X = g.standard_normal((3, 16))
    Ws, Wv = g.standard_normal((8, 16)), g.standard_normal((8, 16))
    Uk, Uv = g.standard_normal((2, 3, 16)), g.standard_normal((2, 3, 16))
    a = grouped.project_grouped(X, Ws, Wv, Uk, Uv, 1)
    b = oracle.project(X, Ws, Wv, Uk, Uv)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x.reshape(y.shape), y, rtol=1e-14)


def test_identical_groups_are_one_basis():
    """G copies of the same shared rows (every group's basis equal) give the
    single-basis oracle's result for every head, paged, to rounding."""
    g = np.random.default_rng(6)
    H, G, d_h, r, ps = 6, 3, 8, 2, 4
    lens = [5, 9]
    pt = np.array([[0, 1, 0], [2, 3, 4]])
    S_K, S_V = g.standard_normal((5, ps, d_h)), g.standard_normal((5, ps, d_h))
    R_K, R_V = g.standard_normal((5, ps, H, r)), g.standard_normal((5, ps, H, r))
    q = g.standard_normal((2, H, d_h))
    BK, BV = g.standard_normal((H, d_h, r)), g.standard_normal((H, d_h, r))
    rep = lambda S: np.repeat(S[:, :, None, :], G, axis=2)
    a = grouped.decode_grouped(q, rep(S_K), rep(S_V), R_K, R_V, BK, BV, pt, lens, ps)
    b = oracle.decode(q, S_K, S_V, R_K, R_V, BK, BV, pt, lens, ps)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-13)


def test_paged_matches_per_request():
    g = np.random.default_rng(5)
    H, G, d_h, r, ps = 4, 2, 8, 2, 4
    lens = [1, 6, 9]
    pt = np.array([[3, 0, 0], [1, 4, 0], [5, 2, 6]])
    pools = [g.standard_normal((7, ps, G, d_h)), g.standard_normal((7, ps, G, d_h)),
             g.standard_normal((7, ps, H, r)), g.standard_normal((7, ps, H, r))]
    q = g.standard_normal((3, H, d_h))
    BK, BV = g.standard_normal((H, d_h, r)), g.standard_normal((H, d_h, r))
    out = grouped.decode_grouped(q, *pools, BK, BV, pt, lens, ps)
    for b, L in enumerate(lens):
        rows = [oracle.gather_rows(p, pt[b], L, ps) for p in pools]
        np.testing.assert_allclose(out[b], grouped.decode_request_grouped(q[b], *rows, BK, BV),
                                   rtol=1e-13)


def test_payload_ratio():
    """(G d_h + H r) / (H d_h) = G/H + r/d_h; G = 1 is the single-basis
    ratio of section 4 (pinned elsewhere), G = H with r = 0 is 1 (MHA)."""
    assert grouped.payload_ratio_grouped(16, 128, 32, 2) == Fraction(3, 8)
    assert grouped.payload_ratio_grouped(16, 128, 48, 1) == Fraction(7, 16)
    assert grouped.payload_ratio_grouped(16, 128, 48, 1) == oracle.payload_ratio(16, 128, 48)
    assert grouped.payload_ratio_grouped(8, 64, 0, 8) == 1


@pytest.mark.parametrize("mutation", ["group_mod", "group_first"])
def test_mutations_fail(monkeypatch, mutation):
    """Planted mistakes in the group mapping fail the pins above."""
    if mutation == "group_mod":
        monkeypatch.setattr(grouped, "group_of", lambda h, H, G: h % G)
    else:
        monkeypatch.setattr(grouped, "group_of", lambda h, H, G: 0)
    with pytest.raises(AssertionError):
        test_zero_query_averages_by_hand()
