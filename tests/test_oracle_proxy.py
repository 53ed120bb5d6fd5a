"""Pins for the oracle's singular proxy and cosine drift (SPA-Cache, "1. Update
identification via singular proxy").  Each check ties the oracle to mathematics
that does not come from the oracle itself: SVD identities, closed-form cosines,
structured projections, and exact special cases."""
import math

import numpy as np
import pytest

from sparse_kv_cache_rank_gb300 import synth


def _rand(shape, seed, scale=1.0):
    return (synth.rng(seed).standard_normal(shape) * scale).astype(np.float32)


# --------------------------------------------------------------------------- SVD / P
def test_full_rank_proxy_cosine_equals_value_cosine(orc):
    """With r = rank(W_V) the proxy cosine is the cosine of the full value states
    (the page's 'full-dimension value identifier'), gain folded in; d != d_kv so a
    wrong side of the SVD cannot even be formed."""
    d, dkv = 48, 32
    w_v = _rand((dkv, d), 1, 0.02)
    gamma = (0.5 + synth.rng(2).random(d)).astype(np.float32)   # non-trivial gain
    P = orc.proxy_matrix(w_v, gamma, dkv)                     # full rank
    assert P.shape == (d, dkv)
    H0 = _rand((1, 16, d), 3)
    H1 = H0 + _rand((1, 16, d), 4, 0.3)
    s0 = H0.astype(np.float64) @ P
    s1, drift = orc.proxy_score(H1, P, s0.astype(np.float32))
    v0 = (H0[0] * gamma) @ w_v.T.astype(np.float64)
    v1 = (H1[0] * gamma) @ w_v.T.astype(np.float64)
    cos_v = (v0 * v1).sum(1) / np.sqrt((v0 * v0).sum(1) * (v1 * v1).sum(1))
    np.testing.assert_allclose(drift[0], 1.0 - cos_v, rtol=2e-4, atol=1e-6)


def test_proxy_energy_and_orthogonality(orc):
    """P^T P = diag(sigma^2) (orthogonal columns scaled by singular values), and at
    full rank trace(P^T P) = ||diag(gamma) W_V^T||_F^2."""
    d, dkv = 40, 24
    w_v = _rand((dkv, d), 5, 0.02)
    gamma = (0.5 + synth.rng(6).random(d)).astype(np.float32)
    A = gamma[:, None].astype(np.float64) * w_v.T.astype(np.float64)
    P = orc.proxy_matrix(w_v, gamma, dkv)
    G = P.T @ P
    off = G - np.diag(np.diag(G))
    assert np.abs(off).max() < 1e-12 * np.abs(G).max()
    assert np.all(np.diff(np.diag(G)) <= 1e-15)                 # descending
    assert math.isclose(np.trace(G), (A * A).sum(), rel_tol=1e-12)


def test_truncation_keeps_the_top_singular_directions(orc):
    """Eckart-Young: the residual of A after projecting onto span(P_r) has spectral
    norm sigma_{r+1}; keeping the bottom directions instead would leave sigma_1."""
    d, dkv, r = 64, 64, 8
    w_v = _rand((dkv, d), 7, 0.02)
    gamma = np.ones(d, np.float32)
    A = w_v.T.astype(np.float64)
    P = orc.proxy_matrix(w_v, gamma, r)
    Q, _ = np.linalg.qr(P)
    resid = A - Q @ (Q.T @ A)
    sig = orc.proxy_singular_values(w_v, gamma)
    assert math.isclose(np.linalg.norm(resid, 2), sig[r], rel_tol=1e-10)
    assert sig[r] < sig[0]


# --------------------------------------------------------------------------- cosine
def test_cosine_special_cases(orc):
    r = 16
    a = _rand((r,), 8)
    b = np.zeros(r, np.float32)
    b[0] = 1.0
    orth = np.zeros(r, np.float32)
    orth[1] = 2.5
    cases = np.stack([a, a, a, b, b, np.zeros(r, np.float32), np.zeros(r, np.float32)])
    other = np.stack([a, 2 * a, -a, orth, -3 * b, np.zeros(r, np.float32), b])
    d = orc.cosine_drift(cases, other)
    assert d[0] == 0.0                          # identical -> exactly 0
    assert abs(d[1]) < 1e-7                     # same direction
    assert abs(d[2] - 2.0) < 1e-7               # antiparallel
    assert abs(d[3] - 1.0) < 1e-7               # orthogonal
    assert abs(d[4] - 2.0) < 1e-7
    assert d[5] == 0.0                          # both zero: nothing moved
    assert d[6] == 1.0                          # one zero


@pytest.mark.parametrize("theta", [1e-3, 0.1, 0.7, 1.5, 2.9])
def test_cosine_known_angle(orc, theta):
    r = 32
    u = np.zeros(r, np.float32)
    v = np.zeros(r, np.float32)
    u[3], u[7] = 1.0, 0.0
    v[3], v[7] = math.cos(theta), math.sin(theta)
    d = orc.cosine_drift(u[None] * 3.0, v[None] * 0.25)[0]
    want = 1.0 - math.cos(theta)
    # inputs are fp32-rounded cos/sin; the drift is then exact to fp32 rounding
    assert abs(d - want) <= 1e-6 * max(1.0, want) + 2e-7


def test_proxy_selection_matrix(orc):
    """P that picks coordinates (c_0 .. c_{r-1}) of h: s_j must equal h[c_j]
    (catches a transposed or mis-strided projection)."""
    B, N, d, r = 2, 5, 12, 4
    cols = [7, 2, 11, 0]
    P = np.zeros((d, r), np.float32)
    for j, c in enumerate(cols):
        P[c, j] = 1.0
    H = _rand((B, N, d), 9)
    cur, _ = orc.proxy_score(H, P, np.ones((B, N, r), np.float32))
    np.testing.assert_array_equal(cur, H[:, :, cols])


def test_proxy_identical_inputs_give_zero_drift(orc):
    """Identical inputs: cosine 1 and drift exactly 0 for every row."""
    sh = synth.TINY
    w = synth.layer_weights(sh, 0)
    P = orc.proxy_matrix(w["w_v"], w["gamma1"], sh.r).astype(np.float32)
    Hp, _, _ = synth.hidden_pair(sh, 0)
    cached, _ = orc.proxy_score(Hp, P, np.ones((sh.B, sh.N, sh.r), np.float32))
    cur, drift = orc.proxy_score(Hp, P, cached)
    np.testing.assert_array_equal(cur, cached)
    assert (drift == 0.0).all()


def test_proxy_scale_invariance(orc):
    """RMSNorm is a positive per-row scale; the drift must not depend on it."""
    d, r = 32, 8
    P = _rand((d, r), 10)
    H0 = _rand((1, 6, d), 11)
    H1 = H0 + _rand((1, 6, d), 12, 0.2)
    c0, _ = orc.proxy_score(H0, P, np.ones((1, 6, r), np.float32))
    _, d1 = orc.proxy_score(H1, P, c0)
    _, d2 = orc.proxy_score(H1 * 4.0, P, c0 * 0.5)
    np.testing.assert_allclose(d1, d2, rtol=1e-6, atol=1e-9)
