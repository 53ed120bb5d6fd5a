"""Attention-distribution drift -- TEST INFRASTRUCTURE ONLY.

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline leg of `bench.py` may import
this module; the product library never imports, links or calls it.

Follows "Polestar: drift-aware cache correction and token commit for efficient diffusion
LLM inference", 2. A (Polestar-Cache), drift measurement: the drift of token i between
consecutive steps is the KL divergence of its attention distributions,
D_i = KL(A_i^t || A_i^{t-1}), and the attention used for it is a proxy attention computed
from compressed representations (same section, sparse updates).

Reading used here (the page gives no formula for A beyond this): the attention
distribution of row i is the softmax over all N rows j of the sequence (bidirectional,
j = i included) of the scaled dot product of proxies, <s_i, s_j> / sqrt(r), where s are
the singular proxies of the rows ("Singular proxies for adaptive caching in diffusion
language models", 1. Update identification via singular proxy); A^t uses the proxies of
the current step and A^{t-1} the cached ones.  Then

    D_i = sum_j A_i^t(j) (ln A_i^t(j) - ln A_i^{t-1}(j)).

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
    out = np.empty(cur.shape[:2])
    for b in range(cur.shape[0]):
        lp = log_softmax_rows(proxy_attention_logits(cur[b]))
        lq = log_softmax_rows(proxy_attention_logits(cached[b]))
        out[b] = (np.exp(lp) * (lp - lq)).sum(axis=-1)
    return out
