"""Attention-distribution drift -- TEST INFRASTRUCTURE ONLY.

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline leg of `bench.py` may import
this module; the product library never imports, links or calls it.

Follows "Polestar: drift-aware cache correction and token commit for efficient diffusion
LLM inference", 2. A (Polestar-Cache), drift measurement: the drift of token i between
consecutive steps is the KL divergence of its attention distributions,
D_i = KL(A_i^t || A_i^{t-1}), and the attention used for it is a proxy attention computed
from compressed representations (same section, sparse updates).

Reading used here (the page gives no formula for A beyond this): the attention
distribution of row i is the softmax, over the other N - 1 rows j != i of the sequence
(bidirectional), of the scaled dot product of proxies <s_i, s_j> / sqrt(r), where s are the
singular proxies of the rows ("Singular proxies for adaptive caching in diffusion language
models", 1. Update identification via singular proxy); A^t uses the proxies of the current
step and A^{t-1} the cached ones.  The row itself is left out because with the same proxy
as query and key its own logit |s_i|^2 / sqrt(r) dwarfs the others and every distribution
would be one-hot on itself.  Then

    D_i = sum_{j != i} A_i^t(j) (ln A_i^t(j) - ln A_i^{t-1}(j)),   D_i = 0 when N = 1.

fp64 throughout; numpy's matmul is the only library step.
"""
from __future__ import annotations

import numpy as np


def log_softmax_rows(x):
    """ln softmax of every row of x, shifted by the row maximum."""
    x = np.asarray(x, dtype=np.float64)
    m = x.max(axis=-1, keepdims=True)
    return x - m - np.log(np.exp(x - m).sum(axis=-1, keepdims=True))


def proxy_attention_logits(S):
    """S [N, r] proxies of one sequence -> [N, N] logits <s_i, s_j> / sqrt(r)."""
    S = np.asarray(S, dtype=np.float64)
    return (S @ S.T) / np.sqrt(S.shape[-1])


def kl_drift(cur, cached):
    """cur, cached [B, N, r] proxies (this step, cached) -> D [B, N] fp64."""
    cur = np.asarray(cur, dtype=np.float64)
    cached = np.asarray(cached, dtype=np.float64)
    if cur.shape != cached.shape or cur.ndim != 3:
        raise ValueError("cur and cached must both be [B, N, r]")
    B, N, _ = cur.shape
    out = np.zeros((B, N))
    if N < 2:
        return out
    off = ~np.eye(N, dtype=bool)
    for b in range(B):
        x = proxy_attention_logits(cur[b])
        y = proxy_attention_logits(cached[b])
        # the N - 1 other rows of every row (row i's own column removed)
        x = x[off].reshape(N, N - 1)
        y = y[off].reshape(N, N - 1)
        lp = log_softmax_rows(x)
        lq = log_softmax_rows(y)
        out[b] = (np.exp(lp) * (lp - lq)).sum(axis=-1)
    return out
