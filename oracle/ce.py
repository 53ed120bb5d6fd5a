"""Confidence extrapolation -- TEST INFRASTRUCTURE ONLY.

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline leg of `bench.py` may import
this module; the product library never imports, links or calls it.

Follows "Efficient diffusion LLMs via temporal-spatial parallel decoding and confidence
extrapolation", 2. Confidence Extrapolation (CE): the confidence of every token is the
noisy observation of a latent (level, velocity) state, filtered like a Kalman filter; the
filter forecasts the near-future confidence with its uncertainty; a risk-aware rule bounds
the look-ahead horizon by the left context already fixed and by a conservative lower bound
of the forecast; a token is committed early when that lower bound exceeds a minimum
threshold.

Reading used here (the page gives the structure, not the equations or constants):
  state x = (l, v), covariance P (2 x 2), constant-velocity model with unit step:
    predict   l- = l + v,  v- = v,  P- = F P F^T + diag(q_l, q_v),  F = [[1, 1], [0, 1]]
    update    S = P-_00 + R,  K = (P-_00, P-_10) / S,  e = c - l-,
              l = l- + K_0 e,  v = v- + K_1 e,  P = (I - K [1 0]) P-
  a token seen for the first time starts at l = c, v = 0, P = diag(R, p_v0) (no update);
  forecast h steps ahead: mean l + h v, variance P_00 + 2 h P_01 + h^2 P_11;
  lower bound LB_h = mean - z sqrt(variance);
  horizon H = min(h_max, number of committed positions left of the token in its block);
  early commit of an undecided token iff LB_h >= c_min for some h in 1 .. H.
fp64 throughout.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class CEParams:
    q_l: float = 1e-3      # process noise of the level
    q_v: float = 1e-3      # process noise of the velocity
    R: float = 1e-2        # observation noise of the confidence
    p_v0: float = 1e-2     # initial velocity variance
    z: float = 1.645       # one-sided 95 % lower bound
    h_max: int = 4         # look-ahead cap
    c_min: float = 0.9     # the static confidence threshold of the commit rule


def init_state(c, prm: CEParams = CEParams()):
    """First observation: l = c, v = 0, P = diag(R, p_v0) -> state [..., 5] (l, v, P00, P01, P11)."""
    c = np.asarray(c, dtype=np.float64)
    st = np.zeros(c.shape + (5,))
    st[..., 0] = c
    st[..., 2] = prm.R
    st[..., 4] = prm.p_v0
    return st


def kalman_step(st, c, prm: CEParams):
    """One predict + update of every state with the observed confidence c."""
    st = np.array(st, dtype=np.float64, copy=True)
    c = np.asarray(c, dtype=np.float64)
    l, v, p00, p01, p11 = (st[..., i] for i in range(5))
    # predict: x- = F x, P- = F P F^T + Q
    lm = l + v
    vm = v
    m00 = p00 + 2 * p01 + p11 + prm.q_l
    m01 = p01 + p11
    m11 = p11 + prm.q_v
    # update with the observation of the level
    S = m00 + prm.R
    k0, k1 = m00 / S, m01 / S
    e = c - lm
    st[..., 0] = lm + k0 * e
    st[..., 1] = vm + k1 * e
    st[..., 2] = (1 - k0) * m00
    st[..., 3] = (1 - k0) * m01
    st[..., 4] = m11 - k1 * m01
    return st


def forecast(st, h):
    """Mean and variance of the confidence h steps ahead."""
    st = np.asarray(st, dtype=np.float64)
    mean = st[..., 0] + h * st[..., 1]
    var = st[..., 2] + 2 * h * st[..., 3] + h * h * st[..., 4]
    return mean, var


def left_coverage(committed):
    """committed [B, M] bool -> number of committed positions left of each position."""
    committed = np.asarray(committed, dtype=bool)
    csum = np.cumsum(committed, axis=-1)
    return csum - committed.astype(np.int64)


def early_commit(st, undecided, committed, prm: CEParams):
    """undecided, committed [B, M] bool -> early [B, M] bool."""
    H = np.minimum(prm.h_max, left_coverage(committed))
    out = np.zeros(np.shape(undecided), dtype=bool)
    for h in range(1, prm.h_max + 1):
        mean, var = forecast(st, h)
        lb = mean - prm.z * np.sqrt(np.maximum(var, 0.0))
        out |= (h <= H) & (lb >= prm.c_min)
    return out & np.asarray(undecided, dtype=bool)


def ce_step(st, seen, c, undecided, committed, prm: CEParams = CEParams()):
    """One step: states of tokens seen before are filtered with c, new ones initialised;
    returns (new state, early-commit decisions)."""
    seen = np.asarray(seen, dtype=bool)
    new = np.where(seen[..., None], kalman_step(st, c, prm), init_state(c, prm))
    return new, early_commit(new, undecided, committed, prm)


def steady_level_variance(q, R):
    """Level-only random walk (v = 0, q_v = 0): the fixed point of the posterior variance,
    P = (P + q) R / (P + q + R)  ->  P = (-q + sqrt(q^2 + 4 q R)) / 2."""
    return (-q + math.sqrt(q * q + 4 * q * R)) / 2
