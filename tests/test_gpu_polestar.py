"""GPU-vs-oracle parity of the drift-aware commit (Polestar, "2. B. Polestar-Commit")
through the C ABI.  Each side carries its own drift history from step to step (fp32 on
the device, fp64 in the oracle): histories within 2e-6 relative (one fp32 rounding of the
sum per step, up to 10 steps), commits equal except where the drift delta lies within
1e-5 of the dynamic threshold (fp32 and fp64 may split that tie)."""
import numpy as np
import pytest

from oracle import polestar as ps
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


@pytest.mark.parametrize("Bq,M,alpha", [(2, 96, 1.0), (1, 1, 1.0), (3, 1000, 4.0), (2, 64, 0.0)])
def test_polestar_commit_parity(B, Bq, M, alpha):
    prm = ps.PolestarParams(alpha=alpha)
    g = synth.rng(2000 + M)
    block = min(M, 32)
    hist = torch.zeros((Bq, M, 2), device="cuda")
    committed = np.zeros((Bq, M), dtype=bool)
    n_commit = 0
    prev = np.zeros((Bq, M, 2))         # the oracle's own history, carried from step to step
    for step in range(10):
        drift = (g.random((Bq, M)) * np.exp(-0.2 * step) + 0.3 * (g.random((Bq, M)) < 0.1)).astype(np.float32)
        conf = g.random((Bq, M)).astype(np.float32)
        suffix = np.zeros((Bq, M), dtype=bool)
        suffix[:, block:] = True
        selected = g.random((Bq, M)) < 0.3
        undecided = ~committed
        c_gpu = B.dllm_polestar_commit(torch.from_numpy(drift).cuda(), torch.from_numpy(conf).cuda(),
                                       _u8(undecided), _u8(suffix), _u8(selected), hist, alpha=alpha,
                                       tau_s=prm.tau_s)
        torch.cuda.synchronize()
        c_ref, hs, hc = ps.commit(drift, conf, undecided, suffix, selected, prev[..., 0], prev[..., 1], prm)
        h_gpu = hist.cpu().numpy().astype(np.float64)
        np.testing.assert_allclose(h_gpu[..., 0], hs, rtol=2e-6, atol=1e-7)
        np.testing.assert_array_equal(h_gpu[..., 1], hc)
        delta = ps.drift_delta(drift, prev[..., 0], prev[..., 1])
        tie = undecided & ~suffix & (prev[..., 1] >= 1) & (np.abs(delta - ps.dynamic_threshold(conf, prm)) < BAND)
        cg = c_gpu.cpu().numpy().astype(bool)
        assert np.array_equal(cg & ~tie, c_ref & ~tie)
        n_commit += int(c_ref.sum())
        prev = np.stack([hs, hc], axis=-1)
        committed |= c_ref
    if M > 8:
        assert n_commit > 0
