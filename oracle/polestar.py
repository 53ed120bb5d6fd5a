"""Drift-aware token commit -- TEST INFRASTRUCTURE ONLY.

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline leg of `bench.py` may import
this module; the product library never imports, links or calls it.

Follows "Polestar: drift-aware cache correction and token commit for efficient diffusion
LLM inference", 2. B (Polestar-Commit):
  * current block: the drift delta of a token, its drift minus the historical mean of its
    drift, signals convergence; the token is committed when the delta exceeds the
    confidence-conditioned threshold tau_d = alpha (tau_s - c)^2;
  * suffix block: when the suffix is among the top drifted positions, suffix tokens are
    committed only at confidence >= tau_s.

Reading used here (the page gives no alpha, tau_s or definition of the history):
  history of token j = the drifts it had at the earlier steps (sum and count);
  delta_j = drift_j - sum_j / count_j, defined once count_j >= 1;
  current-block token:  commit iff undecided and count >= 1 and delta > alpha (tau_s - c)^2;
  suffix token:         commit iff undecided and selected at this step (among the rows the
                        drift score refreshed) and c >= tau_s;
  afterwards every token's history takes this step's drift (sum += drift, count += 1).
fp64 throughout.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class PolestarParams:
    alpha: float = 1.0     # scale of the dynamic threshold
    tau_s: float = 0.9     # high-confidence threshold (the static threshold of the commit rule)


def drift_delta(drift, hist_sum, hist_count):
    """delta = drift - mean of the earlier drifts; nan where there is no history."""
    drift = np.asarray(drift, dtype=np.float64)
    cnt = np.asarray(hist_count, dtype=np.float64)
    with np.errstate(invalid="ignore", divide="ignore"):
        mean = np.where(cnt > 0, np.asarray(hist_sum, dtype=np.float64) / np.where(cnt > 0, cnt, 1), np.nan)
    return drift - mean


def dynamic_threshold(conf, prm: PolestarParams):
    conf = np.asarray(conf, dtype=np.float64)
    return prm.alpha * (prm.tau_s - conf) ** 2


def commit(drift, conf, undecided, suffix, selected, hist_sum, hist_count, prm: PolestarParams = PolestarParams()):
    """All [B, M]; suffix / selected / undecided bool.  Returns (commit [B, M] bool,
    new hist_sum, new hist_count)."""
    drift = np.asarray(drift, dtype=np.float64)
    undecided = np.asarray(undecided, dtype=bool)
    suffix = np.asarray(suffix, dtype=bool)
    selected = np.asarray(selected, dtype=bool)
    cnt = np.asarray(hist_count)
    delta = drift_delta(drift, hist_sum, cnt)
    cur = undecided & ~suffix & (cnt >= 1) & (delta > dynamic_threshold(conf, prm))
    suf = undecided & suffix & selected & (np.asarray(conf, dtype=np.float64) >= prm.tau_s)
    return cur | suf, np.asarray(hist_sum, dtype=np.float64) + drift, cnt + 1
