"""Host-side planning of the tensor-core GEMM, queried through the C ABI without a GPU
(dllm_gemm_plan answers on the host for a given SM count).

* The plans of the LLaDA-8B-shaped layer's projections at 164 gathered rows on a 152-SM
  GB300 are the ones the profiles were measured with (grid, cluster K split, stages).
* For more than 256 tokens, the widths the tile-time model picks on the measured
  projections (Dream-7B-shaped layer and the LLaDA-8B-shaped layer at N = 2048 ... 8192)
  are the measured-fastest ones, except N = 8192 at 100 % down (model 160, measured 224,
  both faster than 256); where the tiles leave a round far from full (O and down at a
  few hundred rows) the model adds a K split.
* Invariants over a grid of shapes, split requests and SM counts: the tile fits the
  tensor-memory and TMA limits, every token row is covered exactly once, K splits leave
  every CTA at least two K blocks, the pipeline has at least two stages and the shared
  memory stays within the per-CTA limit (within half an SM when two CTAs share one).
"""
import os
import shutil

import pytest

SMEM_LIMIT = 232448        # 227 KB of dynamic shared memory per CTA
SMEM_PER_SM = 233472       # 228 KB per SM, 1 KB of it reserved per resident CTA


@pytest.fixture(scope="module")
def B():
    import sparse_kv_cache_rank_gb300 as pkg
    from sparse_kv_cache_rank_gb300 import binding
    if not os.path.exists(binding.LIB_PATH):
        if not shutil.which("nvcc") and not os.path.exists("/usr/local/cuda/bin/nvcc"):
            pytest.skip("nvcc not available to build libdllm.so")
        pkg.build()
    return binding


def test_layer_step_plans_at_164_rows(B):
    """QKV: 96 weight tiles x K split 3 (288 CTAs, two per SM, three stages once the 1 KB
    alignment slack is dropped); O and down: 32 x 4 in clusters of 4 with the whole shared
    memory (one CTA per SM); gate/up: 192 weight tiles, no split, three stages at two CTAs
    per SM.  The 164 rows are staged as 168 (the 8-row swizzle atom) in a 176-column MMA."""
    want = {
        (12288, 4096): dict(splits=3, w_tiles=96, ctas_per_sm=2, stages=3),
        (4096, 4096): dict(splits=4, w_tiles=32, ctas_per_sm=1),
        (24576, 4096): dict(splits=1, w_tiles=192, ctas_per_sm=2, stages=3),
        (4096, 12288): dict(splits=4, w_tiles=32, ctas_per_sm=1),
    }
    for (N_out, K), exp in want.items():
        p = B.dllm_gemm_plan(164, N_out, K, sms=152)
        assert p["BN"] == 176 and p["xrows"] == 168 and p["tok_tiles"] == 1
        for k, v in exp.items():
            assert p[k] == v, (N_out, K, k, p)


def test_few_tiles_get_a_k_split(B):
    """Past 256 rows, O and down (32 weight tiles of the LLaDA-8B-shaped layer) at a few
    hundred rows have fewer tiles than SMs: the width model's K split over a cluster fills
    the GPU (256-288 CTAs at two per SM) instead of leaving 96-192 CTAs to stream all K
    blocks alone (down at 328 rows: 86 -> 45 us on a GB300)."""
    for M, BN, splits, ctas in ((271, 160, 4, 256), (328, 128, 3, 288), (410, 160, 3, 288), (656, 176, 2, 256)):
        for N_out, K in ((4096, 4096), (4096, 12288)):
            p = B.dllm_gemm_plan(M, N_out, K, sms=152)
            assert p["BN"] == BN and p["splits"] == splits and p["ctas_per_sm"] == 2, (M, N_out, K, p)
            assert p["tok_tiles"] * p["w_tiles"] * p["splits"] == ctas


def _proj(d, dq, dkv, F):
    return {"qkv": (dq + 2 * dkv, d), "oproj": (d, dq), "gateup": (2 * F, d), "down": (d, F)}


@pytest.mark.parametrize("M,shape,want", [
    (2624, (3584, 3584, 512, 18944), {"qkv": 176, "oproj": 128, "gateup": 256, "down": 128}),
    (2048, (4096, 4096, 4096, 12288), {"qkv": 256, "oproj": 256, "gateup": 256, "down": 256}),
    (656, (4096, 4096, 4096, 12288), {"qkv": 224, "gateup": 224}),
    (1311, (4096, 4096, 4096, 12288), {"qkv": 224, "oproj": 160, "gateup": 224, "down": 160}),
    (8192, (4096, 4096, 4096, 12288), {"qkv": 256, "oproj": 224, "gateup": 256, "down": 160}),
])
def test_many_token_widths(B, M, shape, want):
    for name, (N_out, K) in _proj(*shape).items():
        if name not in want:
            continue
        p = B.dllm_gemm_plan(M, N_out, K, sms=152)
        assert p["BN"] == want[name], (M, name, p)
        assert p["splits"] == 1 and p["ctas_per_sm"] == 2


MS = [1, 5, 16, 17, 33, 96, 164, 255, 256, 257, 300, 513, 656, 1000, 1311, 2048, 2624, 4096, 8192, 16384]
NS = [32, 96, 128, 512, 2080, 4096, 4608, 12288, 24576, 37888, 152064]
KS = [64, 128, 640, 4096, 18944]


@pytest.mark.parametrize("sms", [152, 148, 132])
@pytest.mark.parametrize("splits", [0, 1, 3, 8])
def test_plan_invariants(B, sms, splits):
    for M in MS:
        for N_out in NS:
            for K in KS:
                for slices in ((0, 1, 2) if splits == 0 else (0,)):
                    if slices == 2 and N_out > 128:
                        continue
                    p = B.dllm_gemm_plan(M, N_out, K, splits=splits, sms=sms, slices=slices)
                    case = (M, N_out, K, splits, sms, slices, p)
                    BN, s, KB = p["BN"], p["splits"], K // 64
                    assert BN % 16 == 0 and 16 <= BN <= 256, case            # MMA N, TMEM columns
                    assert p["xrows"] % 8 == 0 and p["xrows"] <= BN, case      # swizzle atom, TMA box
                    assert (p["tok_tiles"] - 1) * BN < M <= p["tok_tiles"] * BN, case
                    if p["tok_tiles"] == 1:
                        assert p["xrows"] >= M, case
                    else:
                        assert p["xrows"] == BN, case
                    assert p["w_tiles"] == (N_out + 127) // 128, case
                    assert 1 <= s <= 8, case                                   # portable cluster
                    assert s == 1 or KB // s >= 2, case
                    if splits > 0 and not slices:
                        assert s <= splits, case
                    assert p["stages"] >= 2, case
                    assert p["smem"] <= SMEM_LIMIT, case
                    assert p["ctas_per_sm"] * (p["smem"] + 1024) <= SMEM_PER_SM, case


def test_proxy_drift_plan(B):
    """The proxy projection at r = 128, d = 4096.  At 1024 tokens (the LLaDA-8B-shaped
    layer) its slice plan splits K 8 ways over 16 token tiles of 64 rows (128 CTAs, four
    stages each at two CTAs per SM): partials summed by the cosine kernel.  At 16 x 8192 tokens the 1024 token
    tiles of 128 rows fill the GPU without a split, and the drift plan (the same tiles,
    one CTA each, two per SM) computes the drift in the epilogue."""
    p = B.dllm_gemm_plan(1024, 128, 4096, sms=152, slices=1)
    assert (p["BN"], p["splits"], p["tok_tiles"], p["stages"], p["ctas_per_sm"]) == (64, 8, 16, 4, 2)
    p = B.dllm_gemm_plan(16 * 8192, 128, 4096, sms=152, slices=1)
    assert (p["BN"], p["splits"], p["tok_tiles"]) == (128, 1, 1024)
    p = B.dllm_gemm_plan(16 * 8192, 128, 4096, sms=152, slices=2)
    assert (p["BN"], p["splits"], p["tok_tiles"], p["w_tiles"], p["ctas_per_sm"]) == (128, 1, 1024, 1, 2)
    with pytest.raises(B.DllmError):
        B.dllm_gemm_plan(1024, 256, 4096, slices=2)    # the drift needs every feature in one tile
    with pytest.raises(B.DllmError):
        B.dllm_gemm_plan(1024, 128, 4096, slices=3)


def test_plan_rejects_bad_shapes(B):
    with pytest.raises(B.DllmError):
        B.dllm_gemm_plan(16, 128, 100)          # K % 64
    with pytest.raises(B.DllmError):
        B.dllm_gemm_plan(16, 100, 128)          # N_out % 32
    with pytest.raises(B.DllmError):
        B.dllm_gemm_plan(16, 128, 128, sms=0)
    with pytest.raises(B.DllmError):
        B.dllm_gemm_plan(0, 128, 128)
    with pytest.raises(B.DllmError):
        B.dllm_gemm_plan(16, 128, 128, splits=9)
