"""Pins for the oracle's confidence extrapolation ("Efficient diffusion LLMs via
temporal-spatial parallel decoding and confidence extrapolation", 2. Confidence
Extrapolation).  Each check ties `oracle.ce` to something other than itself: the
textbook Kalman gain and Riccati fixed point, the exact tracking of a constant and of a
ramp by a constant-velocity model, hand-computed first steps, and the structure of the
risk-aware decision."""
import math

import numpy as np
import pytest

from oracle import ce
from sparse_kv_cache_rank_gb300 import synth


def test_first_update_by_hand():
    """Second observation after init: P- = F P F^T + Q by hand, gain P-_00/(P-_00 + R),
    posterior by the Joseph-free update."""
    prm = ce.CEParams(q_l=0.01, q_v=0.02, R=0.04, p_v0=0.03)
    st = ce.init_state(np.array([0.5]), prm)
    st2 = ce.kalman_step(st, np.array([0.7]), prm)[0]
    m00 = 0.04 + 0.03 + 0.01
    m01 = 0.03
    m11 = 0.03 + 0.02
    k0, k1 = m00 / (m00 + 0.04), m01 / (m00 + 0.04)
    assert st2[0] == pytest.approx(0.5 + k0 * 0.2, abs=1e-15)
    assert st2[1] == pytest.approx(k1 * 0.2, abs=1e-15)
    assert st2[2] == pytest.approx((1 - k0) * m00, abs=1e-15)
    assert st2[3] == pytest.approx((1 - k0) * m01, abs=1e-15)
    assert st2[4] == pytest.approx(m11 - k1 * m01, abs=1e-15)


def test_level_only_riccati_fixed_point():
    """With q_v = 0 and a zero velocity variance the filter is the scalar random-walk
    filter; its posterior variance converges to (-q + sqrt(q^2 + 4 q R)) / 2."""
    prm = ce.CEParams(q_l=2e-3, q_v=0.0, R=1e-2)
    st = ce.init_state(np.zeros(1), prm)
    st[..., 4] = 0.0   # no velocity uncertainty: the velocity stays 0
    for _ in range(400):
        st = ce.kalman_step(st, np.zeros(1), prm)
    assert st[0, 2] == pytest.approx(ce.steady_level_variance(2e-3, 1e-2), rel=1e-9)
    assert st[0, 4] == 0.0 and st[0, 1] == 0.0


def test_constant_and_ramp_are_tracked():
    """A constant-velocity filter fed exact data: a constant converges to (c, 0), a ramp
    a + b t to level a + b t and velocity b (no steady-state lag)."""
    prm = ce.CEParams()
    st = ce.init_state(np.array([0.3, 0.1]), prm)
    for t in range(1, 300):
        st = ce.kalman_step(st, np.array([0.3, 0.1 + 0.002 * t]), prm)
    assert st[0, 0] == pytest.approx(0.3, abs=1e-9) and abs(st[0, 1]) < 1e-9
    assert st[1, 0] == pytest.approx(0.1 + 0.002 * 299, abs=1e-7)
    assert st[1, 1] == pytest.approx(0.002, abs=1e-8)


def test_covariance_stays_symmetric_positive():
    prm = ce.CEParams()
    g = synth.rng(3)
    st = ce.init_state(g.random(50), prm)
    for _ in range(30):
        st = ce.kalman_step(st, g.random(50), prm)
        det = st[:, 2] * st[:, 4] - st[:, 3] ** 2
        assert np.all(st[:, 2] > 0) and np.all(st[:, 4] > 0) and np.all(det > 0)


def test_forecast_mean_and_variance():
    st = np.array([[0.6, 0.05, 0.01, 0.002, 0.003]])
    mean, var = ce.forecast(st, 3)
    assert mean[0] == pytest.approx(0.75)
    assert var[0] == pytest.approx(0.01 + 6 * 0.002 + 9 * 0.003)


def test_left_coverage_counts():
    committed = np.array([[0, 1, 1, 0, 1, 0, 0, 1]], dtype=bool)
    np.testing.assert_array_equal(ce.left_coverage(committed), [[0, 0, 1, 2, 2, 3, 3, 3]])


def test_decision_structure():
    """No left context -> no early commit; z = 0, h_max = 1 -> commit iff l + v >= c_min;
    raising c_min never adds a commit; only undecided tokens commit."""
    g = synth.rng(5)
    B, M = 3, 32
    st = np.zeros((B, M, 5))
    st[..., 0] = g.uniform(0.5, 1.0, (B, M))
    st[..., 1] = g.uniform(-0.05, 0.15, (B, M))
    st[..., 2] = g.uniform(1e-4, 1e-2, (B, M))
    st[..., 4] = g.uniform(1e-4, 1e-2, (B, M))
    undecided = g.random((B, M)) < 0.7
    committed = ~undecided
    prm = ce.CEParams()
    assert not ce.early_commit(st, undecided, np.zeros((B, M), bool), prm).any()
    p1 = ce.CEParams(z=0.0, h_max=1)
    want = (st[..., 0] + st[..., 1] >= 0.9) & undecided & (ce.left_coverage(committed) >= 1)
    np.testing.assert_array_equal(ce.early_commit(st, undecided, committed, p1), want)
    lo = ce.early_commit(st, undecided, committed, ce.CEParams(c_min=0.8))
    hi = ce.early_commit(st, undecided, committed, ce.CEParams(c_min=0.95))
    assert np.all(hi <= lo)
    assert not (ce.early_commit(st, undecided, committed, prm) & ~undecided).any()


def test_ce_step_initialises_new_tokens():
    prm = ce.CEParams()
    c = np.array([[0.4, 0.8]])
    st, early = ce.ce_step(np.zeros((1, 2, 5)), np.array([[False, False]]), c,
                           np.ones((1, 2), bool), np.zeros((1, 2), bool), prm)
    np.testing.assert_array_equal(st[0, :, 0], [0.4, 0.8])
    assert np.all(st[..., 1] == 0) and np.all(st[..., 2] == prm.R) and np.all(st[..., 4] == prm.p_v0)
    assert not early.any()


def test_lower_bound_closed_form():
    """l = 0.92, v = 0, P00 = 0.01: the 1.645-sigma lower bound one step ahead is
    0.92 - 0.1645 < 0.9, so no early commit; with a small variance (P00 = 1e-4) it is
    0.92 - 0.01645 >= 0.9 and the token commits (one committed position to its left)."""
    prm = ce.CEParams()
    und = np.array([[False, True]])
    com = np.array([[True, False]])
    wide = np.array([[[0.5, 0, 0.01, 0, 0], [0.92, 0.0, 0.01, 0.0, 0.0]]])
    narrow = np.array([[[0.5, 0, 0.01, 0, 0], [0.92, 0.0, 1e-4, 0.0, 0.0]]])
    assert not ce.early_commit(wide, und, com, prm)[0, 1]
    assert ce.early_commit(narrow, und, com, prm)[0, 1]
    mean, var = ce.forecast(wide[0, 1], 1)
    assert mean - prm.z * math.sqrt(var) == pytest.approx(0.92 - 1.645 * 0.1)
