"""Pins for the oracle's attention-distribution drift (Polestar, "2. A. Polestar-Cache",
drift measurement: D_i = KL(A_i^t || A_i^{t-1}) over proxy attention rows).  Every check
ties `oracle.kl` to something other than itself: scipy's softmax / relative entropy on
logits formed by explicit loops, Gibbs' inequality, closed forms (a uniform reference
distribution, three-row sequences) and exact special cases."""
import math

import numpy as np
import pytest
from scipy import special, stats

from oracle import kl as okl
from sparse_kv_cache_rank_gb300 import synth


def _proxies(B, N, r, seed, scale=1.0):
    return synth.rng(seed).standard_normal((B, N, r)) * scale


def _brute(cur, cached):
    """Double loops for the logits, scipy for softmax and the KL terms."""
    B, N, r = cur.shape
    out = np.zeros((B, N))
    for b in range(B):
        for i in range(N):
            others = [j for j in range(N) if j != i]
            x = np.array([sum(cur[b, i, c] * cur[b, j, c] for c in range(r)) for j in others])
            y = np.array([sum(cached[b, i, c] * cached[b, j, c] for c in range(r)) for j in others])
            p = special.softmax(x / math.sqrt(r))
            q = special.softmax(y / math.sqrt(r))
            out[b, i] = special.rel_entr(p, q).sum()
    return out


def test_brute_force_small():
    """Random proxies at N <= 12: equals scipy's relative entropy of the two softmax
    rows over the other rows, so a swapped direction (KL(q || p)), a missing 1/sqrt(r),
    a kept self column or a transposed product fails."""
    cur = _proxies(2, 12, 8, 1, 0.7)
    cached = cur + _proxies(2, 12, 8, 2, 0.4)
    D = okl.kl_drift(cur, cached)
    np.testing.assert_allclose(D, _brute(cur, cached), rtol=1e-10, atol=1e-13)
    # the direction matters on these inputs
    assert np.abs(D - okl.kl_drift(cached, cur)).max() > 1e-3


def test_identical_inputs_give_exact_zero():
    """KL(A || A) = 0: the same proxies at both steps give exactly 0 for every row."""
    cur = _proxies(3, 40, 32, 3)
    assert np.all(okl.kl_drift(cur, cur.copy()) == 0.0)


def test_gibbs_inequality_and_positive_when_different():
    cur = _proxies(2, 64, 32, 4)
    cached = cur.copy()
    cached[:, 5] += _proxies(2, 1, 32, 5)[:, 0]   # one row of each sequence moved
    D = okl.kl_drift(cur, cached)
    assert D.min() >= -1e-12
    assert np.all(D[:, 5] > 1e-3)


def test_uniform_reference_closed_form():
    """Cached proxies all zero: A^{t-1} is uniform over the N - 1 other rows, so
    D_i = ln(N - 1) - H(A_i^t) (entropy from scipy)."""
    N, r = 30, 16
    cur = _proxies(1, N, r, 6)
    D = okl.kl_drift(cur, np.zeros_like(cur))
    x = (cur[0] @ cur[0].T) / math.sqrt(r)
    H = np.array([stats.entropy(special.softmax(np.delete(x[i], i))) for i in range(N)])
    np.testing.assert_allclose(D[0], math.log(N - 1) - H, rtol=1e-10, atol=1e-12)


def test_three_rows_bernoulli_closed_form():
    """N = 3 with collinear proxies s_j = c_j e: row 0 attends to row 1 with
    p = sigmoid(c_0 (c_1 - c_2) / sqrt(r)), so D_0 is the KL of two Bernoulli laws;
    N = 2 leaves one other row, a point mass, and D = 0; N = 1 gives 0."""
    r = 32
    e = np.zeros(r)
    e[3] = 1.0
    c, c2 = (1.3, -0.4, 0.7), (0.9, 0.8, -1.1)
    cur = np.stack([v * e for v in c])[None]
    cached = np.stack([v * e for v in c2])[None]
    sig = lambda z: 1.0 / (1.0 + math.exp(-z))
    p = sig(c[0] * (c[1] - c[2]) / math.sqrt(r))
    q = sig(c2[0] * (c2[1] - c2[2]) / math.sqrt(r))
    want = p * math.log(p / q) + (1 - p) * math.log((1 - p) / (1 - q))
    assert okl.kl_drift(cur, cached)[0, 0] == pytest.approx(want, rel=1e-12, abs=1e-15)
    assert np.all(okl.kl_drift(cur[:, :2], cached[:, :2]) == 0.0)
    assert np.all(okl.kl_drift(cur[:, :1], cached[:, :1]) == 0.0)


def test_row_permutation_equivariance():
    """Relabelling the rows of a sequence (same permutation at both steps) permutes D."""
    cur = _proxies(1, 25, 16, 7)
    cached = cur + _proxies(1, 25, 16, 8, 0.3)
    perm = synth.rng(9).permutation(25)
    D = okl.kl_drift(cur, cached)[0]
    Dp = okl.kl_drift(cur[:, perm], cached[:, perm])[0]
    np.testing.assert_allclose(Dp, D[perm], rtol=1e-12, atol=1e-14)


def test_sequences_are_independent():
    """Each sequence's distribution runs over its own N rows only."""
    cur = _proxies(2, 20, 16, 10)
    cached = cur + _proxies(2, 20, 16, 11, 0.2)
    D = okl.kl_drift(cur, cached)
    np.testing.assert_allclose(D[1], okl.kl_drift(cur[1:], cached[1:])[0], rtol=0, atol=0)
