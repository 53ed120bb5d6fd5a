"""One-time set-up of the singular proxy (SPA-Cache, "Singular proxies for adaptive
caching in diffusion language models", "1. Update identification via singular proxy"):
the value projection is replaced by its rank-r truncated SVD, and each layer input is
projected onto the top-r singular directions.

With the row-vector convention v = RMSNorm(h) W_V^T and the RMSNorm gain folded in,
A = diag(gamma1) W_V^T  [d x d_kv] = U S V^T, and the proxy matrix is P = U_r S_r
[d x r].  The library's proxy kernel takes P^T [r x d] (dllm_proxy_score's `Pt`).

This runs once per layer before any denoising step, never inside a step; the per-step
path (projection, cosine drift, selection, refresh) is the library's kernels.  It uses
the device's dense fp64 factorisations (cuSOLVER through torch.linalg), the way a plain
library product would use cuBLAS.  Only P P^T = U_r S_r^2 U_r^T is defined by the
method -- every drift the kernels compute is invariant to P -> P Q for an orthogonal
r x r Q -- so the signs of the singular vectors are left as the factorisation returns
them.

method="gram" (default): the eigenpairs of the smaller Gram matrix.  For d_kv <= d,
  A^T A = V S^2 V^T, so P = A V_r (= U_r S_r); for d < d_kv, A A^T = U S^2 U^T and
  P = U_r S_r directly.  In fp64 the top-r pairs lose nothing that matters here: the
  Gram squares the condition number, which costs accuracy only in singular values far
  below sigma_1, and those are the ones dropped.
method="svd": the thin SVD of A, fp64.
"""
from __future__ import annotations

import torch

__all__ = ["build_proxy_matrix", "proxy_matrix_f64"]


def proxy_matrix_f64(w_v: torch.Tensor, gamma1: torch.Tensor, r: int, method: str = "gram") -> torch.Tensor:
    """P = U_r S_r of diag(gamma1) W_V^T as an fp64 [d, r] device tensor.

    w_v: [d_kv, d] (nn.Linear layout), gamma1: [d], both CUDA tensors."""
    if not (w_v.is_cuda and gamma1.is_cuda):
        raise ValueError("the proxy set-up runs on the device: pass CUDA tensors")
    d_kv, d = w_v.shape
    if gamma1.shape != (d,):
        raise ValueError(f"gamma1 must be [{d}] (got {tuple(gamma1.shape)})")
    if not 0 < r <= min(d, d_kv):
        raise ValueError(f"rank {r} must be in [1, min(d, d_kv) = {min(d, d_kv)}]")
    A = gamma1.double()[:, None] * w_v.double().t()            # [d, d_kv]
    if method == "svd":
        U, S, _ = torch.linalg.svd(A, full_matrices=False)
        return U[:, :r] * S[:r]
    if method != "gram":
        raise ValueError(f"unknown method {method!r} (use 'gram' or 'svd')")
    if d_kv <= d:
        lam, V = torch.linalg.eigh(A.t() @ A)                  # ascending eigenvalues
        Vr = V[:, -r:].flip(1)                                   # top r, descending
        return A @ Vr
    lam, U = torch.linalg.eigh(A @ A.t())
    top = lam[-r:].flip(0).clamp_min(0.0)
    return U[:, -r:].flip(1) * top.sqrt()


def build_proxy_matrix(w_v: torch.Tensor, gamma1: torch.Tensor, r: int, method: str = "gram",
                       dtype: torch.dtype | None = None) -> torch.Tensor:
    """Pt = P^T [r, d], contiguous, in `dtype` (default: w_v's dtype) -- the `Pt` argument
    of dllm_proxy_score."""
    P = proxy_matrix_f64(w_v, gamma1, r, method)
    return P.t().contiguous().to(dtype or w_v.dtype)
