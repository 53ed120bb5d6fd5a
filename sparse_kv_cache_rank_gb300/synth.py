"""Seeded synthetic inputs shared by the CUDA path, the oracle, the tests and the bench.

This module draws random numbers and converts dtypes; it holds none of the
method's arithmetic (no projection, norm, attention, selection or entropy).
Both sides of every parity check receive the arrays produced here, so a
difference between them can only come from the computation under test.

Workload recipe (restated from the SPA-Cache and EntropyCache pages, see the
configuration docstrings below):
  * weights ~ N(0, 0.02), RMSNorm gains = 1;
  * step t-1 hidden states ~ N(0, 1);
  * step t hidden states = step t-1 + N(0, 0.05) on every row, plus N(0, 0.5)
    on exactly round(0.1 * N) rows per sequence chosen by a seeded permutation;
  * logits for the commit rule ~ N(0, 3) (small configuration);
  * bf16 configurations round every float array to bf16 (round-to-nearest-even)
    and widen it back to fp32, so both sides see identical values.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

__all__ = [
    "LayerShape", "TINY", "LLADA_LAYER", "LLADA_STACK", "DREAM_STACK", "sweep_shapes",
    "rng", "round_bf16", "to_bf16_bits", "from_bf16_bits",
    "layer_weights", "hidden_pair", "hidden_ladder", "drifted", "block_layout", "commit_logits",
]


@dataclasses.dataclass(frozen=True)
class LayerShape:
    """Shape of one bidirectional transformer layer and of its cache."""
    name: str
    B: int            # sequences in the batch
    N: int            # tokens per sequence (prompt + generation)
    d: int            # model width
    n_q: int          # query heads
    n_kv: int         # key/value heads
    hd: int           # head dimension
    F: int            # SwiGLU hidden width
    r: int            # proxy rank
    rho: float        # update ratio (fraction of N refreshed by drift)
    dtype: str        # "f32" or "bf16"
    V: int = 0        # vocabulary (0 = no vocab step in this configuration)
    prompt: int = 0   # prompt tokens (generation starts here)
    block: int = 32   # semi-autoregressive block length
    layers: int = 1
    k_recent: int = 0
    eps: float = 1e-5
    rope_theta: float = 10000.0

    @property
    def d_q(self) -> int:
        return self.n_q * self.hd

    @property
    def d_kv(self) -> int:
        return self.n_kv * self.hd


# Tiny single layer, fp32: seq 256 (128 prompt + 128 masked generation, block 32),
# d=512, 8 heads x 64, FFN 1536, vocab 4096, r=32, 25% update ratio, 8 recent tokens.
TINY = LayerShape("tiny-fp32", B=1, N=256, d=512, n_q=8, n_kv=8, hd=64, F=1536, r=32,
                  rho=0.25, dtype="f32", V=4096, prompt=128, block=32, k_recent=8)

# LLaDA-8B-shaped single layer, bf16: seq 1024 (512 + 512), d=4096, 32 MHA heads x 128,
# FFN 12288, r=128, 16% update ratio.
LLADA_LAYER = LayerShape("llada8b-layer", B=1, N=1024, d=4096, n_q=32, n_kv=32, hd=128,
                         F=12288, r=128, rho=0.16, dtype="bf16", prompt=512)

# Full 32-layer LLaDA-8B-shaped stack: seq 768 (512 prompt + 256 generation), vocab 126464.
LLADA_STACK = LayerShape("llada8b-stack", B=1, N=768, d=4096, n_q=32, n_kv=32, hd=128,
                         F=12288, r=128, rho=0.16, dtype="bf16", V=126464, prompt=512,
                         layers=32)

# Dream-7B-shaped (Qwen2.5-7B layout) stack: batch 8, seq 2048 (1024 + 1024), d=3584,
# 28 query / 4 KV heads x 128, FFN 18944, vocab 152064.
DREAM_STACK = LayerShape("dream7b-stack", B=8, N=2048, d=3584, n_q=28, n_kv=4, hd=128,
                         F=18944, r=128, rho=0.16, dtype="bf16", V=152064, prompt=1024,
                         layers=28)


def sweep_shapes():
    """Long-context sweep on the LLaDA-8B-shaped layer: N x B x update ratio."""
    out = []
    for N in (2048, 4096, 8192):
        for B in (1, 4, 16):
            for rho in (0.05, 0.16, 0.50, 1.00):
                out.append(dataclasses.replace(LLADA_LAYER, name=f"llada8b-N{N}-B{B}-rho{rho}",
                                               N=N, B=B, rho=rho, prompt=N // 2))
    return out


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def round_bf16(x: np.ndarray) -> np.ndarray:
    """fp32 -> nearest bf16 (ties to even) -> fp32. NaN stays NaN."""
    return from_bf16_bits(to_bf16_bits(x))


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    rounded = ((u.astype(np.uint64) + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    return np.where(nan, np.uint16(0x7FC0), rounded).astype(np.uint16)


def from_bf16_bits(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _maybe_round(a: np.ndarray, dtype: str) -> np.ndarray:
    a = a.astype(np.float32)
    return round_bf16(a) if dtype == "bf16" else a


def layer_weights(shape: LayerShape, seed: int, std: float = 0.02) -> dict:
    """Random-init layer weights in nn.Linear layout ([out, in]), fp32 arrays.

    Keys: w_q [d_q, d], w_k [d_kv, d], w_v [d_kv, d], w_o [d, d_q],
    w_g [F, d], w_u [F, d], w_d [d, F], gamma1 [d], gamma2 [d].
    """
    g = rng(seed)
    d, dq, dkv, F = shape.d, shape.d_q, shape.d_kv, shape.F

    def lin(o, i):
        return _maybe_round(g.standard_normal((o, i), dtype=np.float32) * np.float32(std), shape.dtype)

    w = {
        "w_q": lin(dq, d), "w_k": lin(dkv, d), "w_v": lin(dkv, d), "w_o": lin(d, dq),
        "w_g": lin(F, d), "w_u": lin(F, d), "w_d": lin(d, F),
        "gamma1": np.ones(d, np.float32), "gamma2": np.ones(d, np.float32),
    }
    return w


def hidden_pair(shape: LayerShape, seed: int, frac: float = 0.10,
                sigma_all: float = 0.05, sigma_hot: float = 0.5):
    """(H_prev, H_cur, hot_rows): the seeded drift model.

    H_prev ~ N(0,1); H_cur = H_prev + N(0, sigma_all) everywhere plus
    N(0, sigma_hot) on round(frac*N) rows per sequence (seeded permutation).
    hot_rows is a [B, n_hot] int32 array of the perturbed rows (sorted).
    """
    g = rng(seed)
    B, N, d = shape.B, shape.N, shape.d
    h_prev = g.standard_normal((B, N, d), dtype=np.float32)
    h_cur = h_prev + g.standard_normal((B, N, d), dtype=np.float32) * np.float32(sigma_all)
    n_hot = int(round(frac * N))
    hot = np.zeros((B, n_hot), np.int32)
    for b in range(B):
        rows = np.sort(g.permutation(N)[:n_hot]).astype(np.int32)
        hot[b] = rows
        h_cur[b, rows] += g.standard_normal((n_hot, d), dtype=np.float32) * np.float32(sigma_hot)
    return _maybe_round(h_prev, shape.dtype), _maybe_round(h_cur, shape.dtype), hot


def block_layout(shape: LayerShape, seed: int, block_index: int = 0):
    """Current semi-AR block: (masked positions [B, n_masked], recent positions [B, k_recent]).

    The block starts at prompt + block_index*block; k_recent of its positions are
    already decoded (seeded choice) and form the recent history, the rest are masked.
    """
    g = rng(seed)
    start = shape.prompt + block_index * shape.block
    pos = np.arange(start, start + shape.block, dtype=np.int32)
    masked, recent = [], []
    for _ in range(shape.B):
        perm = g.permutation(shape.block)
        rec = np.sort(pos[perm[:shape.k_recent]])
        msk = np.sort(pos[perm[shape.k_recent:]])
        recent.append(rec)
        masked.append(msk)
    return np.stack(masked).astype(np.int32), np.stack(recent).astype(np.int32)


def commit_logits(B: int, M: int, V: int, seed: int, std: float = 3.0) -> np.ndarray:
    """Logits [B, M, V] ~ N(0, std), fp32."""
    g = rng(seed)
    return (g.standard_normal((B, M, V), dtype=np.float32) * np.float32(std)).astype(np.float32)


def hidden_ladder(shape: LayerShape, h_prev: np.ndarray, exclude, seed: int, n_hot: int = 12,
                  sigma_all: float = 0.0, s0: float = 0.02, ratio: float = 1.8) -> np.ndarray:
    """Step-t hidden states with graded drift: h_prev + N(0, sigma_all) on every row, and on
    n_hot rows per sequence (drawn from the rows not in exclude[b], which may hold -1
    padding) an extra N(0, s0 * ratio^j), j = 0 .. n_hot-1.  The moved rows' drifts then
    lie on a geometric ladder, each rung well apart from the next."""
    g = rng(seed)
    B, N, d = shape.B, shape.N, shape.d
    h = h_prev.astype(np.float32) + g.standard_normal((B, N, d), dtype=np.float32) * np.float32(sigma_all)
    for b in range(B):
        ex = set() if exclude is None else {int(i) for i in np.asarray(exclude[b]) if 0 <= i < N}
        cand = np.array([i for i in range(N) if i not in ex], np.int64)
        rows = g.permutation(cand)[:n_hot]
        for j, i in enumerate(rows):
            h[b, i] += g.standard_normal(d, dtype=np.float32) * np.float32(s0 * ratio ** j)
    return _maybe_round(h, shape.dtype)


def drifted(shape: LayerShape, h: np.ndarray, seed: int, frac: float = 0.10,
            sigma_all: float = 0.05, sigma_hot: float = 0.5) -> np.ndarray:
    """The drift model of hidden_pair applied to given states h [B, N, d]: + N(0, sigma_all)
    everywhere, + N(0, sigma_hot) on round(frac * N) rows per sequence (seeded)."""
    g = rng(seed)
    B, N, d = h.shape
    out = h.astype(np.float32) + g.standard_normal((B, N, d), dtype=np.float32) * np.float32(sigma_all)
    n_hot = int(round(frac * N))
    for b in range(B):
        rows = np.sort(g.permutation(N)[:n_hot])
        out[b, rows] += g.standard_normal((n_hot, d), dtype=np.float32) * np.float32(sigma_hot)
    return _maybe_round(out, shape.dtype)
