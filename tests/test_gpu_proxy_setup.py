"""The one-time proxy set-up (SPA-Cache, "1. Update identification via singular proxy":
the top-r singular vectors and values of the value projection, with the RMSNorm gain
folded in) against the oracle's LAPACK SVD (oracle/svd.py), for both of the set-up's
methods, at the LLaDA-8B width (d = d_kv = 4096, r = 128), the Dream-7B shape (d = 3584,
d_kv = 512), and small shapes with d > d_kv and d < d_kv.

What the method defines is P P^T = U_r S_r^2 U_r^T (every drift is invariant to P -> P Q
for an orthogonal Q, so column signs are free): it must match within 1e-4 of its largest
entry, P^T P must be diag(S_r^2), and the cosine drift each P gives on the same seeded
inputs, through the library's fp32 proxy kernel against the oracle's, must match within
the fp32 reduction tolerance.
"""
import functools

import numpy as np
import pytest

from sparse_kv_cache_rank_gb300 import synth
from cases import assert_drift_close, to_dev

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

PPT_RTOL = 1e-4

SHAPES = {"llada": (4096, 4096, 128), "dream": (3584, 512, 128), "narrow-kv": (256, 128, 64),
          "wide-kv": (128, 512, 64)}


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_kv_cache_rank_gb300 import binding
    binding.lib()
    return binding


@functools.lru_cache(maxsize=None)
def _case(name):
    import oracle
    d, d_kv, r = SHAPES[name]
    g = synth.rng(900 + d + d_kv)
    w_v = synth.round_bf16((g.standard_normal((d_kv, d)) * 0.02).astype(np.float32))
    gamma = synth.round_bf16((0.5 + g.random(d)).astype(np.float32))     # a non-trivial gain
    P_o = oracle.proxy_matrix(w_v, gamma, r)                              # fp64 [d, r]
    S = oracle.proxy_singular_values(w_v, gamma)[:r]
    return w_v, gamma, P_o, S


@pytest.mark.parametrize("method", ["gram", "svd"])
@pytest.mark.parametrize("name", list(SHAPES))
def test_proxy_matrix_matches_oracle(B, orc, name, method):
    from sparse_kv_cache_rank_gb300.proxy_setup import build_proxy_matrix, proxy_matrix_f64
    d, d_kv, r = SHAPES[name]
    w_v, gamma, P_o, S = _case(name)
    P_g = proxy_matrix_f64(to_dev(w_v, torch.bfloat16), to_dev(gamma, torch.bfloat16), r, method)
    P_g = P_g.cpu().numpy()
    assert P_g.shape == (d, r)
    G_o = P_o @ P_o.T
    G_g = P_g @ P_g.T
    assert np.abs(G_g - G_o).max() <= PPT_RTOL * np.abs(G_o).max()
    # the columns are the singular directions scaled by the singular values, in order
    PtP = P_g.T @ P_g
    np.testing.assert_allclose(np.diag(PtP), S ** 2, rtol=1e-6)
    assert np.abs(PtP - np.diag(np.diag(PtP))).max() <= 1e-6 * S[0] ** 2
    # the drift each P yields on the same seeded inputs (fp32 path of the proxy kernel)
    sh = synth.LayerShape("p", B=1, N=96, d=d, n_q=1, n_kv=1, hd=64, F=64, r=r, rho=0.1, dtype="f32")
    H_prev, H_cur, _ = synth.hidden_pair(sh, 901)
    P32_o = P_o.astype(np.float32)
    pc, _ = orc.proxy_score(H_prev, P32_o, np.ones((1, sh.N, r), np.float32))
    _, drift_o = orc.proxy_score(H_cur, P32_o, pc)
    Pt = build_proxy_matrix(to_dev(w_v, torch.bfloat16), to_dev(gamma, torch.bfloat16), r, method,
                            dtype=torch.float32)
    ones = torch.ones((1, sh.N, r), device="cuda")
    pc_g, _ = B.dllm_proxy_score(to_dev(H_prev), Pt, ones)
    _, drift_g = B.dllm_proxy_score(to_dev(H_cur), Pt, pc_g)
    assert_drift_close(drift_g.cpu().numpy(), drift_o)


def test_proxy_setup_refuses_host_tensors():
    from sparse_kv_cache_rank_gb300.proxy_setup import proxy_matrix_f64
    with pytest.raises(ValueError):
        proxy_matrix_f64(torch.zeros((8, 16)), torch.ones(16), 4)
