"""Pins for the oracle's selection (SPA-Cache "1. Update identification via singular
proxy": lowest similarity first; "2. Adaptive budget allocation": per-layer budget;
EntropyCache "How EntropyCache works" step 3: masked and recent tokens always
recomputed).  Checked by exhaustive search on tiny inputs and by special cases."""
import itertools
import math

import numpy as np
import pytest

from sparse_kv_cache_rank_gb300 import synth


def _exhaustive(drift, forced, k, min_drift):
    """Best subset by exhaustive search: among all subsets of the eligible rows of the
    allowed size, the one whose (drift desc, index asc) key list is lexicographically
    largest -- a different algorithm from the oracle's repeated max extraction."""
    N = len(drift)
    fset = {int(f) for f in forced if 0 <= f < N}
    elig = [i for i in range(N) if i not in fset and drift[i] > min_drift]
    size = min(k, N - len(fset), len(elig))
    best, best_key = (), None
    for sub in itertools.combinations(elig, size):
        key = sorted(((float(drift[i]), -i) for i in sub), reverse=True)
        if best_key is None or key > best_key:
            best, best_key = sub, key
    return sorted(fset | set(best))


@pytest.mark.parametrize("seed", range(12))
def test_select_matches_exhaustive_search(orc, seed):
    g = synth.rng(100 + seed)
    N = int(g.integers(1, 11))
    # draw from a small value set so that equal drifts (ties) happen often
    drift = g.choice(np.array([0.0, 1e-7, 0.1, 0.3, 0.3, 0.5, 0.9], np.float32), size=N)
    F = int(g.integers(0, 4))
    forced = g.integers(-2, N + 2, size=F).astype(np.int32)
    k = int(g.integers(0, N + 2))
    idx, cnt = orc.select_topk(drift[None], forced[None] if F else None, k, 1e-6)
    want = _exhaustive(drift, forced, k, 1e-6)
    assert cnt[0] == len(want)
    assert list(idx[0, :cnt[0]]) == want
    assert (idx[0, cnt[0]:] == -1).all()


def test_select_edge_cases(orc):
    N = 20
    drift = np.linspace(0.5, 0.01, N, dtype=np.float32)[None]
    forced = np.array([[3, 3, -1, 19, 25]], np.int32)       # duplicate and padding
    idx, cnt = orc.select_topk(drift, forced, 0, 1e-6)        # k = 0 -> forced only
    assert list(idx[0, :cnt[0]]) == [3, 19]
    idx, cnt = orc.select_topk(drift, forced, N, 1e-6)        # everything
    assert cnt[0] == N and list(idx[0, :N]) == list(range(N))
    idx, cnt = orc.select_topk(drift, None, 4, 1e-6)          # no forced set
    assert list(idx[0, :cnt[0]]) == [0, 1, 2, 3]
    z = np.zeros((2, N), np.float32)                          # identical inputs
    idx, cnt = orc.select_topk(z, None, 5, 1e-6)
    assert (cnt == 0).all()
    nan = np.full((1, N), np.nan, np.float32)
    nan[0, 7] = 0.2
    idx, cnt = orc.select_topk(nan, None, 5, 1e-6)
    assert list(idx[0, :cnt[0]]) == [7]


def test_select_is_per_sequence(orc):
    drift = np.array([[0.1, 0.9, 0.2, 0.3], [0.9, 0.1, 0.8, 0.0]], np.float32)
    idx, cnt = orc.select_topk(drift, None, 2, 1e-6)
    assert list(idx[0, :2]) == [1, 3] and list(idx[1, :2]) == [0, 2]


def test_drift_ranks_perturbed_rows_first(orc):
    """On the seeded drift model (10% of rows moved by N(0,0.5), the rest by
    N(0,0.05)) the proxy drift must put every strongly moved row into a 16% budget;
    choosing the least drifted rows instead would select none of them."""
    sh = synth.LayerShape("mid", B=1, N=512, d=512, n_q=4, n_kv=4, hd=128, F=64, r=64,
                          rho=0.16, dtype="bf16")
    w = synth.layer_weights(sh, 3)
    P = orc.proxy_matrix(w["w_v"], w["gamma1"], sh.r).astype(np.float32)
    Hp, Hc, hot = synth.hidden_pair(sh, 3)
    cached, _ = orc.proxy_score(Hp, P, np.zeros((1, sh.N, sh.r), np.float32))
    _, drift = orc.proxy_score(Hc, P, cached)
    k = orc.budget(sh.rho, sh.N)
    idx, cnt = orc.select_topk(drift, None, k, 1e-6)
    chosen = set(idx[0, :cnt[0]].tolist())
    assert set(hot[0].tolist()) <= chosen
    assert drift[0, hot[0]].min() > 10 * np.median(drift[0])


def test_budget_schedule(orc):
    # configuration budgets: 25% of 256 and 16% of 1024 and 16% of 2048
    assert orc.budget(0.25, 256) == 64
    assert orc.budget(0.16, 1024) == 164
    assert orc.budget(0.16, 2048) == 328
    assert orc.budget(0.0, 100) == 0
    assert orc.budget(1e-9, 100) == 1
    assert orc.budget(1.0, 100) == 100
    # piecewise Gaussian: peak 0.30 at layer 16, 0.05 floor, sigma 6 layers
    assert orc.rho(16) == pytest.approx(0.30, abs=1e-15)
    assert orc.rho(0) == pytest.approx(0.05 + 0.25 * math.exp(-256 / 72), rel=1e-14)
    assert orc.rho(10) == pytest.approx(orc.rho(22), rel=1e-14)            # symmetric
    assert orc.rho(10, sigma_left=3.0) < orc.rho(22, sigma_left=3.0)       # piecewise
    vals = [orc.rho(l) for l in range(32)]
    assert max(vals) == vals[16] and min(vals) == vals[0]
    ks = [orc.budget(v, 768) for v in vals]
    assert ks[0] == 44 and ks[16] == 231
