"""Pins for the oracle's vocabulary step: top-1 confidence and predictive entropy
(TSPD "Input features"), the maximum entropy of the newly decoded tokens and the
full/partial decision (EntropyCache "How EntropyCache works", steps 2-3), and the
static confidence-threshold commit (Polestar "1. Problem definition")."""
import math

import numpy as np
import pytest
import scipy.special
import scipy.stats

from sparse_kv_cache_rank_gb300 import synth


@pytest.mark.parametrize("V", [2, 7, 4096, 126464])
def test_uniform_distribution(orc, V):
    am, pm, H = orc.vocab_stats(np.zeros((1, 2, V), np.float32))
    assert (am == 0).all()                                   # lowest id on ties
    np.testing.assert_allclose(pm, 1.0 / V, rtol=1e-6)
    np.testing.assert_allclose(H, math.log(V), rtol=1e-6)


def test_dominant_logit(orc):
    V = 4096
    l = synth.rng(1).standard_normal((1, 3, V)).astype(np.float32)
    l[0, 0, 17] += 50.0
    l[0, 1, 4095] += 50.0
    l[0, 2, 0] += 50.0
    am, pm, H = orc.vocab_stats(l)
    assert list(am[0]) == [17, 4095, 0]
    assert (pm > 1 - 1e-6).all() and (pm <= 1.0).all()
    assert (H < 1e-6).all()


@pytest.mark.parametrize("m,a", [(1, 3.0), (5, 1.0), (3, -2.0), (100, 0.5)])
def test_two_level_closed_form(orc, m, a):
    V = 1000
    l = np.zeros((1, 1, V), np.float32)
    hi = np.arange(V - m, V)                                 # high tokens at the end
    l[0, 0, hi] = a
    am, pm, H = orc.vocab_stats(l)
    z = m * math.exp(a) + (V - m)
    p_hi, p_lo = math.exp(a) / z, 1.0 / z
    want_H = -(m * p_hi * math.log(p_hi) + (V - m) * p_lo * math.log(p_lo))
    assert math.isclose(H[0, 0], want_H, rel_tol=1e-6)
    assert math.isclose(pm[0, 0], max(p_hi, p_lo), rel_tol=1e-6)
    assert am[0, 0] == (V - m if a > 0 else 0)


@pytest.mark.parametrize("seed", range(6))
def test_small_vocab_against_scipy(orc, seed):
    g = synth.rng(200 + seed)
    V = int(g.integers(2, 17))
    l = (g.standard_normal((4, V)) * 3).astype(np.float32)
    am, pm, H = orc.vocab_stats(l[None])
    p = scipy.special.softmax(l.astype(np.float64), axis=-1)
    np.testing.assert_allclose(H[0], scipy.stats.entropy(p, axis=-1), rtol=1e-6)
    np.testing.assert_allclose(pm[0], p.max(-1), rtol=1e-6)
    np.testing.assert_array_equal(am[0], np.argmax(l, -1))


def test_commit_rule_cases(orc):
    B, M = 4, 5
    am = np.arange(B * M, dtype=np.int32).reshape(B, M) + 100
    pm = np.array([[0.95, 0.2, 0.9, 0.89, 0.1],      # 0 and 2 (inclusive threshold)
                   [0.3, 0.5, 0.5, 0.1, 0.2],        # none: highest -> row 1 (lowest of tie)
                   [0.99, 0.99, 0.99, 0.99, 0.99],   # all, but row 3 invalid
                   [0.1, 0.1, 0.1, 0.1, 0.1]],       # no valid rows
                  np.float32)
    ent = np.array([[0.3, 5.0, 2.5, 0.1, 0.1],
                    [1.0, 2.0, 7.0, 0.5, 0.5],
                    [0.1, 0.2, 2.0, 9.0, 0.4],
                    [3.0, 3.0, 3.0, 3.0, 3.0]], np.float32)
    valid = np.ones((B, M), np.uint8)
    valid[2, 3] = 0
    valid[3] = 0
    tok, E, full = orc.commit_rule(am, pm, ent, valid, 0.9, 2.0)
    assert list(np.where(tok[0] >= 0)[0]) == [0, 2] and tok[0, 0] == 100 and tok[0, 2] == 102
    assert list(np.where(tok[1] >= 0)[0]) == [1]
    assert list(np.where(tok[2] >= 0)[0]) == [0, 1, 2, 4]
    assert (tok[3] == -1).all()
    np.testing.assert_array_equal(E, np.array([2.5, 2.0, 2.0, 0.0], np.float32))
    # E > tau -> full refresh; E == tau stays partial
    np.testing.assert_array_equal(full, [1, 0, 0, 0])


def test_commit_entropy_composite(orc):
    B, M, V = 2, 24, 4096
    l = synth.commit_logits(B, M, V, 3)
    l[0, 5] *= 10.0                                         # one confident row
    valid = np.ones((B, M), np.uint8)
    valid[1, 10:] = 0
    tok, conf, ent, E, full = orc.commit_entropy(l, valid)
    am, pm, H = orc.vocab_stats(l)
    assert (conf[1, 10:] == 0).all() and (ent[1, 10:] == 0).all() and (tok[1, 10:] == -1).all()
    t2, E2, f2 = orc.commit_rule(am, pm, H, valid)
    np.testing.assert_array_equal(tok, t2)
    np.testing.assert_array_equal(E, E2)


def test_lmhead_one_hot_rows(orc):
    """W_lm rows are unit vectors e_v: logits[m, v] = RMSNorm(h_m)[v] * gamma[v]."""
    M, d = 3, 16
    h = synth.rng(4).standard_normal((M, d)).astype(np.float32)
    gamma = (0.5 + synth.rng(5).random(d)).astype(np.float32)
    W = np.eye(d, dtype=np.float32)[::-1].copy()           # row v = e_{d-1-v}
    out = orc.lmhead(h, gamma, W, eps=1e-5)
    xn = h / np.sqrt((h.astype(np.float64) ** 2).mean(-1, keepdims=True) + 1e-5) * gamma
    np.testing.assert_allclose(out, xn[:, ::-1], rtol=1e-6, atol=1e-7)
