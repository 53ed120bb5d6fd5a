"""Shared helpers for the GPU parity tests: seeded cases (inputs from
sparse_kv_cache_rank_gb300.synth, expected values from the oracle) and the
comparison metrics."""
from __future__ import annotations

import dataclasses

import numpy as np

from sparse_kv_cache_rank_gb300 import synth

# tolerances: selection and commit decisions exact outside a 1e-5 near-tie band, fp32
# reductions within 1e-4 relative, bf16 layer outputs within 2e-2 of the largest
# reference value with cosine >= 0.999
FP32_REDUCTION_RTOL = 1e-4      # drift, entropy, confidence, fp32 proxies
BF16_MAX_REL = 2e-2             # bf16 layer outputs: max |err| / max |ref|
BF16_MIN_COS = 0.999
F32_MAX_REL = 1e-4              # fp32 layer outputs on the CUDA cores
F32_MIN_COS = 0.999999
TIE_BAND = 1e-5                 # selection / commit decisions within this band are near-ties


def torch_dtype(shape):
    import torch
    return torch.bfloat16 if shape.dtype == "bf16" else torch.float32


def to_dev(a, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def to_np(t):
    import torch
    return t.detach().to(torch.float32).cpu().numpy() if t.dtype.is_floating_point else t.cpu().numpy()


def normwise_rel(x, ref):
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.abs(ref).max()
    return float(np.abs(x - ref).max() / (den if den > 0 else 1.0))


def cosine(x, ref):
    x = np.asarray(x, np.float64).ravel()
    ref = np.asarray(ref, np.float64).ravel()
    n = np.linalg.norm(x) * np.linalg.norm(ref)
    return float(x @ ref / n) if n > 0 else 1.0


def assert_close_layer(x, ref, dtype: str, what: str):
    rel, cs = normwise_rel(x, ref), cosine(x, ref)
    if dtype == "bf16":
        assert rel <= BF16_MAX_REL and cs >= BF16_MIN_COS, f"{what}: rel {rel:.3e} cos {cs:.6f}"
    else:
        assert rel <= F32_MAX_REL and cs >= F32_MIN_COS, f"{what}: rel {rel:.3e} cos {cs:.8f}"
    return rel, cs


def assert_update_close(out, ref_out, h_in, dtype: str, what: str, h_in_ref=None):
    """The layer's update (output minus input).  A bf16 output carries the rounding
    of the whole residual sum, so the update is compared against the reference output
    rounded the same way, and the max error may include one bf16 ulp of |output|.
    h_in_ref: the reference side's own input when it differs from the GPU's (a deeper
    layer of a chained step); default h_in."""
    from sparse_kv_cache_rank_gb300 import synth
    ref = synth.round_bf16(ref_out) if dtype == "bf16" else ref_out
    du = np.asarray(out, np.float64) - h_in
    dr = np.asarray(ref, np.float64) - (h_in if h_in_ref is None else h_in_ref)
    cs = cosine(du, dr)
    err = np.abs(du - dr).max()
    if dtype == "bf16":
        # one ulp for the output's rounding, one more for the inputs' own when they differ
        ulp = 2.0 ** (np.floor(np.log2(np.abs(ref).max())) - 7) * (1 if h_in_ref is None else 2)
        bound = BF16_MAX_REL * np.abs(dr).max() + ulp
        assert cs >= BF16_MIN_COS and err <= bound, f"{what}: err {err:.3e} > {bound:.3e} or cos {cs:.6f}"
    else:
        bound = F32_MAX_REL * np.abs(dr).max()
        assert cs >= F32_MIN_COS and err <= bound, f"{what}: err {err:.3e} > {bound:.3e} or cos {cs:.8f}"


def assert_drift_close(gpu, ref):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(gpu - ref)
    bound = FP32_REDUCTION_RTOL * np.abs(ref) + 1e-7
    bad = err > bound
    assert not bad.any(), (f"{bad.sum()} drifts off: worst rel "
                           f"{(err / np.maximum(np.abs(ref), 1e-30)).max():.3e}")


def check_selection_band(idx, cnt, drift_ref, forced, k):
    """GPU selection vs the oracle's drift: counts equal, every row above the k-th
    drift by more than TIE_BAND selected, none below it by more than TIE_BAND."""
    B, N = drift_ref.shape
    for b in range(B):
        sel = set(idx[b, :cnt[b]].tolist())
        fset = set()
        if forced is not None:
            fset = {int(p) for p in forced[b] if 0 <= p < N}
        assert fset <= sel
        elig = [i for i in range(N) if i not in fset and drift_ref[b, i] > 1e-6]
        take = min(k, N - len(fset), len(elig))
        assert cnt[b] == len(fset) + take
        if take == 0 or take == len(elig):
            continue
        order = sorted(elig, key=lambda i: (-drift_ref[b, i], i))
        kth = drift_ref[b, order[take - 1]]
        for i in elig:
            if drift_ref[b, i] > kth + TIE_BAND:
                assert i in sel, f"row {i} drift {drift_ref[b, i]} > kth {kth} not selected"
            if drift_ref[b, i] < kth - TIE_BAND:
                assert i not in sel, f"row {i} drift {drift_ref[b, i]} < kth {kth} selected"


def match_selection(g_idx, g_cnt, drift_ref, o_idx, o_cnt, forced, k):
    """GPU selection against the oracle's own (each side selects on its own drift): equal
    counts, the near-tie band rule, and per sequence the rows both sides chose plus the
    rows only one side chose (which the band rule has already confined to the near-ties
    of the k-th drift).  -> list of (common, gpu_only, oracle_only) sorted index arrays."""
    np.testing.assert_array_equal(g_cnt, o_cnt)
    check_selection_band(g_idx, g_cnt, drift_ref, forced, k)
    out = []
    for b in range(len(g_cnt)):
        gs = set(g_idx[b, :g_cnt[b]].tolist())
        os_ = set(o_idx[b, :o_cnt[b]].tolist())
        out.append((np.array(sorted(gs & os_), np.int64), np.array(sorted(gs - os_), np.int64),
                    np.array(sorted(os_ - gs), np.int64)))
    return out


def softmax_stats_bound(logits_ref, delta):
    """How far top-1 confidence and entropy may move when every logit of a row moves by at
    most delta (derived on the path l + t e, |e| <= delta, t in [0, 1]):
      ln p_k moves by <= 2 delta, so |d p_max| <= p_max (e^{2 delta} - 1);
      dH/dt = -sum_k p_k (l_k - lbar) e_k, and along the path p_k stays within e^{+-2 delta}
      of its start and |l_k - lbar| within 2 delta + (e^{2 delta} - 1) m of it, so
      |d H| <= delta e^{2 delta} (e^{2 delta} m + 2 delta),  m = sum_k p_k |l_k - lbar|.
    -> (conf bound, entropy bound), arrays over the rows of logits_ref [..., V]."""
    l = np.asarray(logits_ref, np.float64)
    z = l - l.max(-1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(-1, keepdims=True)
    lbar = (p * l).sum(-1, keepdims=True)
    m = (p * np.abs(l - lbar)).sum(-1)
    e2 = np.exp(2 * delta)
    return p.max(-1) * (e2 - 1), delta * e2 * (e2 * m + 2 * delta)


@dataclasses.dataclass
class LayerCase:
    shape: synth.LayerShape
    w: dict
    P: np.ndarray           # [d, r] fp32 (dtype-rounded)
    H_prev: np.ndarray
    H_cur: np.ndarray
    hot: np.ndarray
    K0: np.ndarray          # caches before the step (dtype-rounded)
    V0: np.ndarray
    O0: np.ndarray
    pc0: np.ndarray         # cached proxies [B, N, r]


def layer_case(orc, shape: synth.LayerShape, seed: int, consistent: bool = True,
               svd_proxy: bool = True) -> LayerCase:
    """Inputs of one refresh step.  consistent=True builds the caches with the oracle's
    full forward on H_prev (small shapes); otherwise caches are seeded random values of
    the same scale (any cache content is a valid input of the refresh)."""
    w = synth.layer_weights(shape, seed)
    H_prev, H_cur, hot = synth.hidden_pair(shape, seed + 1)
    rnd = synth.round_bf16 if shape.dtype == "bf16" else (lambda a: a.astype(np.float32))
    if svd_proxy:
        P = orc.proxy_matrix(w["w_v"], w["gamma1"], shape.r)
    else:
        g = synth.rng(seed + 2)
        P = g.standard_normal((shape.d, shape.r)) * (0.02 * np.sqrt(shape.d_kv / shape.r))
    P = rnd(P.astype(np.float32))
    if consistent:
        L = orc.Layer(w, shape.n_q, shape.n_kv, shape.hd, eps=shape.eps, rope_theta=shape.rope_theta)
        K0, V0, O0 = orc.layer_full(L, H_prev)
    else:
        g = synth.rng(seed + 3)
        sc = 0.02 * np.sqrt(shape.d)
        K0 = g.standard_normal((shape.B, shape.N, shape.d_kv), dtype=np.float32) * np.float32(sc)
        V0 = g.standard_normal((shape.B, shape.N, shape.d_kv), dtype=np.float32) * np.float32(sc)
        O0 = g.standard_normal((shape.B, shape.N, shape.d), dtype=np.float32)
    K0, V0, O0 = rnd(K0), rnd(V0), rnd(O0)
    pc0, _ = orc.proxy_score(H_prev, P, np.ones((shape.B, shape.N, shape.r), np.float32))
    return LayerCase(shape, w, P, H_prev, H_cur, hot, K0, V0, O0, pc0)


def forced_rows(shape: synth.LayerShape, seed: int):
    """Forced set: the current block's masked positions plus the recent decoded ones."""
    if shape.k_recent == 0 and shape.V == 0:
        return None
    masked, recent = synth.block_layout(shape, seed)
    return np.concatenate([masked, recent], axis=1).astype(np.int32)
