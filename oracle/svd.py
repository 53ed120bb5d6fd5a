"""Proxy matrix of the singular proxy -- oracle side, TEST INFRASTRUCTURE ONLY.

SPA-Cache ("Singular proxies for adaptive caching in diffusion language
models", "1. Update identification via singular proxy"): the value projection
is replaced by its truncated SVD, keeping the top-r singular vectors and
values, and each input state is projected into that rank-r subspace.

Reading taken here (row-vector convention, v = xn W_V^T with xn = RMSNorm(h)):
A = diag(gamma1) W_V^T  [d x d_kv] = U S V^T;  P = U_r S_r  [d x r].
Then h P V_r^T = h A_r is the rank-r value state of h with the norm gain folded
in; because V_r has orthonormal columns, cosines of h P equal cosines of h A_r,
and RMSNorm's positive per-row scale cancels in the cosine.
"""
from __future__ import annotations

import numpy as np


def _a_matrix(w_v, gamma1):
    w_v = np.asarray(w_v, dtype=np.float64)
    g = np.asarray(gamma1, dtype=np.float64)
    return g[:, None] * w_v.T          # [d, d_kv]


def proxy_matrix(w_v, gamma1, r: int) -> np.ndarray:
    """P = U_r S_r of diag(gamma1) W_V^T, fp64 LAPACK SVD, returned as fp64 [d, r]."""
    A = _a_matrix(w_v, gamma1)
    U, S, _ = np.linalg.svd(A, full_matrices=False)
    if r > S.shape[0]:
        raise ValueError(f"rank {r} exceeds min(d, d_kv) = {S.shape[0]}")
    return U[:, :r] * S[:r]


def proxy_singular_values(w_v, gamma1) -> np.ndarray:
    """All singular values of diag(gamma1) W_V^T, descending."""
    return np.linalg.svd(_a_matrix(w_v, gamma1), compute_uv=False)
