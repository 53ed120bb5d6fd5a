"""GPU-vs-oracle parity of confidence extrapolation ("Efficient diffusion LLMs via
temporal-spatial parallel decoding and confidence extrapolation", 2. Confidence
Extrapolation) through the C ABI.

Every step feeds both sides the same previous state (the device's, read back), so the
comparison is of one fp32 predict + update against fp64: states within 1e-5 relative +
1e-6 absolute (a handful of fp32 operations on values of order 1).  Early-commit
decisions are bit-exact except where a lower bound lies within 1e-5 of c_min (the two
precisions may decide such a tie differently); those positions are checked to be
undecided tokens with enough left context.
"""
import numpy as np
import pytest

from oracle import ce
from sparse_kv_cache_rank_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

BAND = 1e-5


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_kv_cache_rank_gb300 import binding
    binding.lib()
    binding.check_status(reset=True)
    return binding


def _u8(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def _near_tie(st, undecided, committed, prm):
    """Positions where some lower bound within the horizon is within BAND of c_min."""
    H = np.minimum(prm.h_max, ce.left_coverage(committed))
    near = np.zeros(undecided.shape, dtype=bool)
    for h in range(1, prm.h_max + 1):
        mean, var = ce.forecast(st, h)
        lb = mean - prm.z * np.sqrt(np.maximum(var, 0.0))
        near |= (h <= H) & (np.abs(lb - prm.c_min) < BAND)
    return near & undecided


@pytest.mark.parametrize("Bq,M,h_max", [(3, 40, 4), (1, 32, 4), (2, 1024, 6), (4, 1, 4), (2, 77, 0)])
def test_ce_steps_parity(B, Bq, M, h_max):
    prm = ce.CEParams(h_max=h_max)
    g = synth.rng(1000 + M + h_max)
    # confidence trajectories: a rising logistic per token with noise, clipped to [0, 1]
    rate = g.uniform(0.05, 0.6, (Bq, M))
    mid = g.uniform(0, 12, (Bq, M))
    state = torch.zeros((Bq, M, 5), device="cuda")
    seen = np.zeros((Bq, M), dtype=bool)
    committed = np.zeros((Bq, M), dtype=bool)
    n_early = 0
    st_o = np.zeros((Bq, M, 5))         # the oracle's own state, carried from step to step
    for step in range(14):
        c = 1 / (1 + np.exp(-rate * (step - mid))) + 0.03 * g.standard_normal((Bq, M))
        c = np.clip(c, 0, 1).astype(np.float32)
        undecided = ~committed
        early = B.dllm_ce_step(torch.from_numpy(c).cuda(), _u8(seen), _u8(undecided), _u8(committed), state,
                               q_l=prm.q_l, q_v=prm.q_v, R=prm.R, p_v0=prm.p_v0, z=prm.z,
                               h_max=prm.h_max, c_min=prm.c_min)
        torch.cuda.synchronize()
        st_ref, early_ref = ce.ce_step(st_o, seen, c, undecided, committed, prm)
        st_o = st_ref
        st_gpu = state.cpu().numpy().astype(np.float64)
        np.testing.assert_allclose(st_gpu, st_ref, rtol=1e-5, atol=1e-6)
        e_gpu = early.cpu().numpy().astype(bool)
        tie = _near_tie(st_ref, undecided, committed, prm)
        assert np.array_equal(e_gpu & ~tie, early_ref & ~tie)
        assert not (e_gpu & ~undecided).any()
        n_early += int(early_ref.sum())
        # the block advances: early commits plus the static rule on the observed confidence
        committed |= early_ref | (c >= prm.c_min)
        seen[:] = True
    if h_max > 0 and M > 8:
        assert n_early > 0   # the trajectories do exercise early commits


def test_ce_degenerate(B):
    """No left context or h_max = 0: never early; unseen tokens are initialised."""
    Bq, M = 2, 64
    c = torch.full((Bq, M), 0.99, device="cuda")
    state = torch.zeros((Bq, M, 5), device="cuda")
    z = _u8(np.zeros((Bq, M)))
    one = _u8(np.ones((Bq, M)))
    early = B.dllm_ce_step(c, z, one, z, state)
    assert not early.any().item()
    st = state.cpu().numpy()
    assert np.all(st[..., 0] == np.float32(0.99)) and np.all(st[..., 1] == 0)
    assert np.all(st[..., 2] == np.float32(1e-2)) and np.all(st[..., 4] == np.float32(1e-2))
    early = B.dllm_ce_step(c, one, one, one, state, h_max=0)
    assert not early.any().item()
