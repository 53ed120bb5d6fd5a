"""Cluster-granular proxy -- TEST INFRASTRUCTURE ONLY.

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline leg of `bench.py` may import
this module; the product library never imports, links or calls it.

Follows "Polestar: drift-aware cache correction and token commit for efficient diffusion
LLM inference", 2. A (Polestar-Cache), local window and clustering / sparse updates: the
hidden states of a local window are clustered with spherical k-means, the residuals are
quantised with NVFP4 into a compressed proxy, and each step the top-k drifted clusters are
refreshed.

Readings used here (the page names the steps, not their equations):
  spherical k-means (Lloyd): u_i = x_i / |x_i| (0 for a zero row); a_i = argmax_k <u_i, c_k>
    (lowest k on ties); c_k = normalise(sum_{a_i = k} u_i), an empty cluster (or a zero
    sum) keeps its centroid; `iters` rounds of assignment then update, and a final
    assignment to the returned centroids;
  residual r_i = x_i - |x_i| c_{a_i} (what the direction of the centroid does not carry);
  NVFP4: blocks of 16 consecutive elements of a row; a per-tensor fp32 scale g;
    block scale s_b = E4M3(amax_b / (6 g)) and element code E2M1(x / (s_b g)) (code 0 when
    s_b = 0), both rounded to nearest even with saturation (E2M1 magnitudes
    {0, .5, 1, 1.5, 2, 3, 4, 6}; E4M3 finite maximum 448, smallest subnormal 2^-9); the
    divisions are taken in fp32, the precision of the device's conversion;
    dequantised value = E2M1 value * E4M3 value * g;
  cluster drift d_k = 1 - cos(c_k^t, c_k^{t-1}) (the SPA identifier at cluster granularity);
    the k_c clusters with the largest drift (lower index on ties) are refreshed: their
    member rows, ascending.
"""
from __future__ import annotations

import numpy as np

E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


# --------------------------------------------------------------------------- k-means
def _unit_rows(X):
    n = np.linalg.norm(X, axis=-1, keepdims=True)
    return np.where(n > 0, X / np.where(n > 0, n, 1), 0.0)


def assign(X, C):
    """X [N, D], C [K, D] unit centroids -> argmax cosine (lowest index on ties)."""
    sims = _unit_rows(np.asarray(X, np.float64)) @ np.asarray(C, np.float64).T
    return np.argmax(sims, axis=1)


def spherical_kmeans(X, C0, iters: int):
    """X [N, D], C0 [K, D] (normalised here) -> (assignment [N], centroids [K, D])."""
    X = np.asarray(X, np.float64)
    U = _unit_rows(X)
    C = _unit_rows(np.asarray(C0, np.float64))
    for _ in range(iters):
        a = np.argmax(U @ C.T, axis=1)
        for k in range(C.shape[0]):
            s = U[a == k].sum(axis=0)
            n = np.linalg.norm(s)
            if n > 0:
                C[k] = s / n
    return np.argmax(U @ C.T, axis=1), C


def residuals(X, C, a):
    X = np.asarray(X, np.float64)
    return X - np.linalg.norm(X, axis=1, keepdims=True) * np.asarray(C, np.float64)[a]


# --------------------------------------------------------------------------- rounding
def e2m1_round(v):
    """Nearest E2M1 value (between two equally near ones, the even code), saturated at
    +-6, sign kept (a negative input that rounds to zero is -0, code 8); returns
    (value, code = sign << 3 | magnitude index)."""
    v = np.asarray(v, dtype=np.float64)
    mag = np.minimum(np.abs(v), 6.0)
    d = np.abs(mag[..., None] - E2M1_GRID)
    tied = d == d.min(axis=-1, keepdims=True)
    codes = np.arange(8)
    idx = np.argmin(np.where(tied, codes % 2, 2), axis=-1)   # adjacent grid codes differ in parity
    sign = np.signbit(v)
    val = np.where(sign, -E2M1_GRID[idx], E2M1_GRID[idx])
    return val, (idx + np.where(sign, 8, 0)).astype(np.uint8)


def _e4m3_values():
    vals = []
    for code in range(0x7F):   # 0x7F is NaN in the E4M3 "fn" variant
        e, m = code >> 3, code & 7
        vals.append(m / 8 * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7))
    return np.array(vals)


E4M3_VALUES = _e4m3_values()   # codes 0 .. 126 ascending, 448 = code 126


def e4m3_round(v):
    """Nearest non-negative E4M3 value (ties to the even code), saturated at 448;
    returns (value, code)."""
    v = np.minimum(np.asarray(v, dtype=np.float64), 448.0)
    d = np.abs(v[..., None] - E4M3_VALUES)
    best = d.min(axis=-1, keepdims=True)
    tied = d == best
    codes = np.arange(E4M3_VALUES.size)
    idx = np.argmin(np.where(tied, codes % 2, 2), axis=-1)   # even code among the tied ones
    return E4M3_VALUES[idx], idx.astype(np.uint8)


# --------------------------------------------------------------------------- NVFP4
def nvfp4_quantize(R, g):
    """R [rows, D] (D % 16 == 0), g > 0 -> (codes [rows, D] uint8 in 0..15, scale codes
    [rows, D/16] uint8).  Divisions in fp32."""
    R = np.asarray(R, dtype=np.float32)
    rows, D = R.shape
    blk = R.reshape(rows, D // 16, 16)
    g32 = np.float32(g)
    amax = np.abs(blk).max(axis=-1)
    s_in = (amax / (np.float32(6.0) * g32)).astype(np.float32)
    s_val, s_code = e4m3_round(s_in)
    s32 = s_val.astype(np.float32)
    denom = (s32 * g32).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q_in = np.where(denom[..., None] > 0, blk / np.where(denom[..., None] > 0, denom[..., None], 1),
                        np.float32(0)).astype(np.float32)
    _, codes = e2m1_round(q_in)
    codes = np.where(denom[..., None] > 0, codes, 0).astype(np.uint8)
    return codes.reshape(rows, D), s_code


def nvfp4_dequantize(codes, s_code, g):
    codes = np.asarray(codes)
    rows, D = codes.shape
    mag = E2M1_GRID[codes & 7]
    val = np.where(codes & 8, -mag, mag)
    s = E4M3_VALUES[np.asarray(s_code)]
    return (val.reshape(rows, D // 16, 16) * s[..., None] * float(np.float32(g))).reshape(rows, D)


# --------------------------------------------------------------------------- selection
def cluster_drift(C_now, C_prev):
    C_now, C_prev = np.asarray(C_now, np.float64), np.asarray(C_prev, np.float64)
    na, nb = np.linalg.norm(C_now, axis=-1), np.linalg.norm(C_prev, axis=-1)
    dot = (C_now * C_prev).sum(-1)
    out = np.where((na > 0) & (nb > 0), 1 - dot / np.where((na > 0) & (nb > 0), na * nb, 1), 0.0)
    out = np.where((na > 0) != (nb > 0), 1.0, out)
    return np.clip(out, 0.0, 2.0)


def select_clusters(C_now, C_prev, a, kc: int):
    """-> (rows ascending, chosen clusters ascending)."""
    d = cluster_drift(C_now, C_prev)
    order = sorted(range(d.size), key=lambda k: (-d[k], k))
    chosen = sorted(order[:max(0, min(kc, d.size))])
    rows = [i for i in range(len(a)) if a[i] in set(chosen)]
    return np.array(rows, dtype=np.int64), np.array(chosen, dtype=np.int64)
