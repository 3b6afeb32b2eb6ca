"""Pins of the oracle's joint key RMSNorm (reading note "Low-Rank Key Value
Attention", section 8), each tied to something other than the oracle: keys
worked by hand, the note's expansion of d_h n^2, scale invariance, RMSNorm
written as k sqrt(d_h) / |k| on the multi-query reduction, the note's warning
that separate normalisation turns the key, and planted mistakes."""
import math

import numpy as np
import pytest
from scipy.special import softmax

import oracle
from oracle import norm as N


def _case(T=7, H=3, d_h=8, r=2, seed=0):
    g = np.random.default_rng(seed)
    return (g.standard_normal((H, d_h)), g.standard_normal((T, d_h)), g.standard_normal((T, d_h)),
            g.standard_normal((T, H, r)), g.standard_normal((T, H, r)),
            g.standard_normal((H, d_h, r)) / math.sqrt(r), g.standard_normal((H, d_h, r)) / math.sqrt(r))


@pytest.mark.parametrize("s,z,B,want", [
    # k = (3, 0) + 1 * (0, 4) = (3, 4): mean square 25/2, no cross term
    ([3.0, 0.0], [1.0], [[0.0], [4.0]], 1.0 / math.sqrt(12.5)),
    # k = (1, 2) + 1 * (3, 1) = (4, 3): |s|^2 = 5, cross 2 (3 + 2) = 10, |B z|^2 = 10
    ([1.0, 2.0], [1.0], [[3.0], [1.0]], 1.0 / math.sqrt(12.5)),
    # k = (1, -1, 2, 0) + (1, 1, 0, 2) = (2, 0, 2, 2) with z = (1, 1), B columns (1,0,0,1), (0,1,0,1)
    ([1.0, -1.0, 2.0, 0.0], [1.0, 1.0], [[1, 0], [0, 1], [0, 0], [1, 1]], 1.0 / math.sqrt(3.0)),
])
def test_inv_norm_by_hand(s, z, B, want):
    S, Z, Bm = np.array([s]), np.array([z]), np.array(B, np.float64)
    assert N.inv_norm(S, Z, Bm, 0.0)[0] == pytest.approx(want, rel=1e-15)
    assert N.inv_norm_expanded(S, Z, Bm, 0.0)[0] == pytest.approx(want, rel=1e-15)
    eps = 0.25
    assert N.inv_norm(S, Z, Bm, eps)[0] == pytest.approx(1 / math.sqrt(1 / want ** 2 + eps), rel=1e-15)


def test_expansion_matches_direct():
    q, SK, SV, RK, RV, BK, BV = _case(T=30, H=4, d_h=16, r=5, seed=1)
    for h in range(4):
        np.testing.assert_allclose(N.inv_norm_expanded(SK, RK[:, h], BK[h], 1e-3),
                                   N.inv_norm(SK, RK[:, h], BK[h], 1e-3), rtol=1e-13)


def test_scale_invariance():
    """With eps = 0 a key's scale drops out; with eps > 0 it does not."""
    q, SK, SV, RK, RV, BK, BV = _case(seed=2)
    a = N.decode_request_norm(q, SK, SV, RK, RV, BK, BV, 0.0)
    b = N.decode_request_norm(q, SK * 7.5, SV, RK * 7.5, RV, BK, BV, 0.0)
    np.testing.assert_allclose(a, b, rtol=1e-12)
    c = N.decode_request_norm(q, SK * 0.01, SV, RK * 0.01, RV, BK, BV, 1.0)
    assert np.abs(a - c).max() > 1e-3


def test_multi_query_reduction_against_norm_formula():
    """Zero private factors: every head attends the shared keys scaled to
    root mean square one, k sqrt(d_h) / |k| (eps = 0)."""
    q, SK, SV, RK, RV, BK, BV = _case(T=9, d_h=8, seed=3)
    out = N.decode_request_norm(q, SK, SV, RK * 0, RV * 0, BK, BV, 0.0)
    Kn = SK * math.sqrt(8) / np.linalg.norm(SK, axis=1, keepdims=True)
    for h in range(q.shape[0]):
        np.testing.assert_allclose(out[h], softmax(Kn @ q[h] / math.sqrt(8)) @ SV, rtol=1e-12)


def test_joint_differs_from_separate():
    """Normalising the shared and private parts each by its own norm turns
    the key (the note's warning): outputs differ from the joint scheme."""
    q, SK, SV, RK, RV, BK, BV = _case(seed=4)
    joint = N.decode_request_norm(q, SK, SV, RK, RV, BK, BV, 0.0)
    sep = np.empty_like(joint)
    for h in range(q.shape[0]):
        P = RK[:, h] @ BK[h].T
        K = N.rms_normalise(SK, 0.0) + N.rms_normalise(P, 0.0)
        V = oracle.expand_head(SV, RV[:, h], BV[h])
        sep[h] = oracle.attend(q[h], K, V)
    assert np.abs(joint - sep).max() > 1e-2


def test_factored_equals_materialised():
    for seed, (T, H, d_h, r) in enumerate([(5, 2, 4, 1), (12, 3, 8, 3), (40, 2, 16, 6)]):
        args = _case(T, H, d_h, r, seed=10 + seed)
        np.testing.assert_allclose(N.decode_request_norm(*args, 1e-5),
                                   N.decode_request_norm_factored(*args, 1e-5), rtol=1e-12)


def test_paged_decode_with_stored_norms():
    g = np.random.default_rng(5)
    H, d_h, r, ps = 2, 8, 2, 4
    lens = [1, 5, 9]
    pt = np.array([[3, 0, 0], [1, 4, 0], [5, 2, 6]])
    pools = [g.standard_normal((7, ps, d_h)), g.standard_normal((7, ps, d_h)),
             g.standard_normal((7, ps, H, r)), g.standard_normal((7, ps, H, r))]
    q = g.standard_normal((3, H, d_h))
    BK, BV = g.standard_normal((H, d_h, r)), g.standard_normal((H, d_h, r))
    NK = N.key_norms(pools[0].reshape(-1, d_h), pools[2].reshape(-1, H, r), BK, 1e-6).reshape(7, ps, H)
    out = N.decode_norm(q, *pools, BK, BV, NK, pt, lens, ps)
    for b, L in enumerate(lens):
        rows = [oracle.gather_rows(p, pt[b], L, ps) for p in pools]
        np.testing.assert_allclose(out[b], N.decode_request_norm(q[b], *rows, BK, BV, 1e-6),
                                   rtol=1e-12)


@pytest.mark.parametrize("mutation", ["no_cross", "sqrt_dh", "no_eps"])
def test_mutations_fail(monkeypatch, mutation):
    orig = N.inv_norm_expanded

    def bad(S, R_h, B_h, eps):
        S, Z, B = (np.asarray(x, np.float64) for x in (S, R_h, B_h))
        d_h = S.shape[1]
        cross = 0.0 if mutation == "no_cross" else 2.0 * np.einsum("td,dr,tr->t", S, B, Z)
        sq = np.sum(S * S, axis=1) + cross + np.einsum("tr,dr,de,te->t", Z, B, B, Z)
        sq = sq + (0.0 if mutation == "no_eps" else d_h * eps)
        return 1.0 / np.sqrt(sq / (math.sqrt(d_h) if mutation == "sqrt_dh" else d_h))

    monkeypatch.setattr(N, "inv_norm_expanded", bad)
    failed = False
    for chk in (lambda: test_inv_norm_by_hand([1.0, 2.0], [1.0], [[3.0], [1.0]], 1 / math.sqrt(12.5)),
                test_expansion_matches_direct):
        try:
            chk()
        except AssertionError:
            failed = True
    assert failed
