"""GPU-vs-oracle parity of the attention-distribution drift (Polestar, "2. A.
Polestar-Cache", drift measurement: D_i = KL(A_i^t || A_i^{t-1}) over row-granular
proxy attention) through the C ABI.

Tolerance (fp32 on the device against the fp64 oracle on the same fp32 proxies): a
score x_ij = <s_i, s_j> / sqrt(r) carries an error of about eps |s_i| |s_j| (an r-term
fp32 dot product, random-walk accumulation, times the 1/sqrt(r) scale).  Under score
errors dx, dy, D moves by sum_j |q_j - p_j| |dy_j| + sum_j p_j |x_j - y_j - E_p(x - y)| |dx_j|,
and the two log-partition sums add about 2 log2(N) eps.  Each row may differ by 16 times
that bound plus 1e-4 of its value.  Identical proxies must give exactly 0.
"""
import math

import numpy as np
import pytest

from oracle import kl as okl
from sparse_kv_cache_rank_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

EPS32 = 2.0 ** -24


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_kv_cache_rank_gb300 import binding
    binding.lib()
    binding.check_status(reset=True)
    return binding


def _drifted(Bq, N, r, seed, noise=0.05, hot_frac=0.1, hot=0.5):
    """Cached proxies ~ N(0, 1); this step's = cached + small noise on every row and a
    larger move on a fraction of the rows (the drift model of the layer inputs)."""
    g = synth.rng(seed)
    cached = g.standard_normal((Bq, N, r))
    cur = cached + noise * g.standard_normal((Bq, N, r))
    n_hot = int(round(hot_frac * N))
    for b in range(Bq):
        rows = g.permutation(N)[:n_hot]
        cur[b, rows] += hot * g.standard_normal((n_hot, r))
    return cur.astype(np.float32), cached.astype(np.float32)


def _tolerance(cur, cached):
    """Per-row bound of the module docstring, from the oracle's own distributions."""
    Bq, N, r = cur.shape
    tol = np.zeros((Bq, N))
    if N < 2:
        return tol + 16 * EPS32
    off = ~np.eye(N, dtype=bool)
    for b in range(Bq):
        s, t = cur[b].astype(np.float64), cached[b].astype(np.float64)
        x = okl.proxy_attention_logits(s)[off].reshape(N, N - 1)
        y = okl.proxy_attention_logits(t)[off].reshape(N, N - 1)
        p = np.exp(okl.log_softmax_rows(x))
        q = np.exp(okl.log_softmax_rows(y))
        d = x - y
        dev = np.abs(d - (p * d).sum(1, keepdims=True))
        ns, nt = np.linalg.norm(s, axis=1), np.linalg.norm(t, axis=1)
        dx = EPS32 * ns * ns.max()
        dy = EPS32 * nt * nt.max()
        tol[b] = 16 * (dy * np.abs(q - p).sum(1) + dx * (p * dev).sum(1) + (2 * math.log2(N) + 1) * EPS32)
    return tol


def _check(gpu, ref, tol):
    err = np.abs(gpu - ref)
    bad = err > tol + 1e-4 * np.abs(ref)
    assert not bad.any(), (f"{bad.sum()} rows off; worst err {err.max():.3e} "
                           f"(tol {tol.ravel()[err.argmax()]:.3e}, ref {ref.ravel()[err.argmax()]:.3e})")


# several query / key tiles, ragged tails (a last tile of one key), one and several
# proxy chunks, clusters of 1 .. 8 key slices
@pytest.mark.parametrize("Bq,N,r", [(1, 64, 32), (2, 200, 64), (3, 129, 128), (1, 333, 160),
                                    (2, 65, 32), (1, 1024, 128), (1, 3, 32)])
def test_kl_drift_parity(B, Bq, N, r):
    cur, cached = _drifted(Bq, N, r, 100 + N + r)
    D = B.dllm_kl_drift(torch.from_numpy(cur).cuda(), torch.from_numpy(cached).cuda())
    torch.cuda.synchronize()
    ref = okl.kl_drift(cur, cached)
    _check(D.cpu().numpy().astype(np.float64), ref, _tolerance(cur, cached))
    assert D.min().item() >= -_tolerance(cur, cached).max() - 1e-12


def test_kl_drift_identical_inputs_exact_zero(B):
    cur, _ = _drifted(2, 300, 128, 7)
    t = torch.from_numpy(cur).cuda()
    D = B.dllm_kl_drift(t, t.clone())
    assert (D == 0).all().item()


@pytest.mark.parametrize("N", [1, 2])
def test_kl_drift_degenerate_sizes(B, N):
    """One row: no other row to attend to; two rows: a point mass on the other row."""
    cur, cached = _drifted(2, N, 64, 8, hot_frac=1.0)
    D = B.dllm_kl_drift(torch.from_numpy(cur).cuda(), torch.from_numpy(cached).cuda())
    assert (D == 0).all().item()


def test_kl_drift_uniform_reference(B):
    """Cached proxies all zero: D_i = ln(N - 1) - H(A_i^t)."""
    cur, _ = _drifted(1, 257, 64, 9)
    cached = np.zeros_like(cur)
    D = B.dllm_kl_drift(torch.from_numpy(cur).cuda(), torch.from_numpy(cached).cuda()).cpu().numpy()
    ref = okl.kl_drift(cur, cached)
    _check(D.astype(np.float64), ref, _tolerance(cur, cached))


def test_kl_drift_selects_the_moved_rows(B):
    """At the layer's shape (N = 1024, r = 128) the top-k of the KL drift, taken by
    dllm_select_topk on the device, equals the oracle's top-k up to rows inside the
    tolerance band of the k-th value, and holds every strongly moved row."""
    N, r, k = 1024, 128, 164
    cur, cached = _drifted(1, N, r, 10)
    D = B.dllm_kl_drift(torch.from_numpy(cur).cuda(), torch.from_numpy(cached).cuda())
    idx, cnt = B.dllm_select_topk(D, None, k)
    torch.cuda.synchronize()
    sel = set(idx[0, :cnt[0]].cpu().tolist())
    ref = okl.kl_drift(cur, cached)[0]
    band = _tolerance(cur, cached)[0].max() + 1e-4 * ref.max()
    order = np.argsort(-ref, kind="stable")
    kth = ref[order[k - 1]]
    assert int(cnt[0]) == k
    for i in range(N):
        if ref[i] > kth + band:
            assert i in sel, f"row {i} KL {ref[i]:.4e} > k-th {kth:.4e} not selected"
        if ref[i] < kth - band:
            assert i not in sel, f"row {i} KL {ref[i]:.4e} < k-th {kth:.4e} selected"
    moved = np.where(np.abs(cur[0] - cached[0]).max(1) > 0.6)[0]
    assert set(moved.tolist()) <= sel
