"""Pins for the oracle's drift-aware commit (Polestar, "2. B. Polestar-Commit"): the delta
against a brute-force mean of the stored drift history, closed forms of the dynamic
threshold alpha (tau_s - c)^2, and the structure of the two rules."""
import numpy as np
import pytest

from oracle import polestar as ps
from sparse_kv_cache_rank_gb300 import synth


def test_history_is_the_mean_of_earlier_drifts():
    """Running (sum, count) over 9 steps gives delta = drift - mean(earlier drifts),
    compared with the explicit mean of the stored list."""
    g = synth.rng(1)
    B, M = 2, 17
    hs, hc = np.zeros((B, M)), np.zeros((B, M), dtype=np.int64)
    past = [[[] for _ in range(M)] for _ in range(B)]
    for _ in range(9):
        d = g.random((B, M))
        delta = ps.drift_delta(d, hs, hc)
        for b in range(B):
            for j in range(M):
                if past[b][j]:
                    assert delta[b, j] == pytest.approx(d[b, j] - sum(past[b][j]) / len(past[b][j]), abs=1e-14)
                else:
                    assert np.isnan(delta[b, j])
                past[b][j].append(d[b, j])
        _, hs, hc = ps.commit(d, np.zeros((B, M)), np.zeros((B, M), bool), np.zeros((B, M), bool),
                              np.zeros((B, M), bool), hs, hc)


def test_threshold_closed_forms():
    prm = ps.PolestarParams(alpha=2.0, tau_s=0.9)
    assert ps.dynamic_threshold(0.9, prm) == 0.0
    assert ps.dynamic_threshold(0.5, prm) == pytest.approx(2.0 * 0.16)
    assert ps.dynamic_threshold(1.0, prm) == pytest.approx(2.0 * 0.01)   # symmetric square


def test_current_block_rule():
    """c = tau_s: commit iff delta > 0; a token without history never commits; a larger
    alpha never adds commits; decided tokens never commit."""
    prm = ps.PolestarParams()
    d = np.array([[0.30, 0.10, 0.50, 0.50]])
    hs = np.array([[0.20, 0.20, 0.0, 0.40]])
    hc = np.array([[1, 1, 0, 1]])
    conf = np.full((1, 4), 0.9)
    und = np.ones((1, 4), bool)
    no = np.zeros((1, 4), bool)
    c, _, _ = ps.commit(d, conf, und, no, no, hs, hc, prm)
    np.testing.assert_array_equal(c, [[True, False, False, True]])
    g = synth.rng(2)
    d, hs, conf = g.random((3, 40)), g.random((3, 40)), g.random((3, 40))
    hc = g.integers(0, 3, (3, 40))
    und = g.random((3, 40)) < 0.8
    c1, _, _ = ps.commit(d, conf, und, np.zeros_like(und), np.zeros_like(und), hs, hc, ps.PolestarParams(alpha=0.5))
    c2, _, _ = ps.commit(d, conf, und, np.zeros_like(und), np.zeros_like(und), hs, hc, ps.PolestarParams(alpha=3.0))
    assert np.all(c2 <= c1)
    assert not (c1 & ~und).any() and not (c1 & (hc == 0)).any()
    # explicit formula, element by element
    want = und & (hc >= 1) & (d - np.where(hc > 0, hs / np.maximum(hc, 1), 0) > 0.5 * (0.9 - conf) ** 2)
    np.testing.assert_array_equal(c1, want)


def test_suffix_rule():
    """Suffix tokens: only when selected and at confidence >= tau_s (inclusive), whatever
    their delta."""
    prm = ps.PolestarParams()
    conf = np.array([[0.95, 0.9, 0.89, 0.99]])
    sel = np.array([[True, True, True, False]])
    suf = np.ones((1, 4), bool)
    d = np.zeros((1, 4))
    hs, hc = np.ones((1, 4)), np.ones((1, 4))
    c, _, _ = ps.commit(d, conf, np.ones((1, 4), bool), suf, sel, hs, hc, prm)
    np.testing.assert_array_equal(c, [[True, True, False, False]])
