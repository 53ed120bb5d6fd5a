"""GPU-vs-oracle parity of the cluster-granular proxy (Polestar, "2. A. Polestar-Cache",
local window and clustering) through the C ABI.

* k-means: assignments equal wherever the oracle's best cosine beats the second by more
  than 1e-4 (well-separated clusters: all rows); centroids and row norms within 1e-5.
* residuals: within 1e-5 of max |x| (one fp32 multiply-add per element).
* NVFP4: codes and block scales bit-exact on the same fp32 inputs (both sides decide in
  fp32, the device conversion's precision), including zero blocks, exact midpoints,
  negative values that round to zero, saturated scales and subnormal scales; the
  dequantised values bit-exact too (code x scale is exact, one rounding by g).
* selection: the same rows and counts when the k-th cluster drift is not within 1e-5 of
  the next one.
"""
import numpy as np
import pytest

from oracle import cluster as cl
from sparse_kv_cache_rank_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_kv_cache_rank_gb300 import binding
    binding.lib()
    binding.check_status(reset=True)
    return binding


def _clustered(Bq, N, D, K, seed, noise=0.3):
    g = synth.rng(seed)
    dirs = g.standard_normal((Bq, K, D))
    dirs /= np.linalg.norm(dirs, axis=-1, keepdims=True)
    lab = g.integers(0, K, (Bq, N))
    X = np.take_along_axis(dirs, lab[..., None], axis=1) + noise * g.standard_normal((Bq, N, D)) / np.sqrt(D)
    X *= g.uniform(0.5, 3.0, (Bq, N, 1))
    C0 = dirs + 0.5 * g.standard_normal((Bq, K, D)) / np.sqrt(D)
    return X.astype(np.float32), C0.astype(np.float32)


@pytest.mark.parametrize("Bq,N,D,K,iters", [(2, 96, 256, 8, 4), (1, 300, 4096, 16, 3), (3, 33, 64, 5, 0)])
def test_kmeans_residual_parity(B, Bq, N, D, K, iters):
    X, C0 = _clustered(Bq, N, D, K, 100 + N)
    Xd = torch.from_numpy(X).cuda()
    Cd = torch.from_numpy(C0.copy()).cuda()
    a, xn = B.dllm_spherical_kmeans(Xd, Cd, iters)
    R = B.dllm_cluster_residual(Xd, Cd, a, xn)
    torch.cuda.synchronize()
    for b in range(Bq):
        a_ref, C_ref = cl.spherical_kmeans(X[b], C0[b], iters)
        U = X[b] / np.linalg.norm(X[b], axis=1, keepdims=True)
        sims = np.sort(U.astype(np.float64) @ C_ref.T, axis=1)
        clear = sims[:, -1] - sims[:, -2] > 1e-4
        assert clear.mean() > 0.95
        np.testing.assert_array_equal(a[b].cpu().numpy()[clear], a_ref[clear])
        np.testing.assert_allclose(Cd[b].cpu().numpy(), C_ref, atol=1e-5)
        np.testing.assert_allclose(xn[b].cpu().numpy(), np.linalg.norm(X[b].astype(np.float64), axis=1), rtol=1e-6)
        # residuals against the oracle's own assignment, on the rows whose assignment is clear
        R_ref = cl.residuals(X[b], C_ref, a_ref)
        assert np.abs(R[b].cpu().numpy()[clear] - R_ref[clear]).max() <= 1e-5 * np.abs(X[b]).max()


def _unpack(codes):
    c = codes.cpu().numpy()
    out = np.empty((c.shape[0], c.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = c & 15
    out[:, 1::2] = c >> 4
    return out


def test_nvfp4_codes_bit_exact(B):
    g = synth.rng(7)
    rows, D = 64, 256
    # blocks spanning many binades (subnormal and saturated E4M3 scales among them)
    R = g.standard_normal((rows, D // 16, 16)) * np.exp2(g.integers(-30, 12, (rows, D // 16, 1)))
    R[0, 0] = 0.0                                                        # zero block
    s = 2.0 ** -4
    R[1, 0] = np.array([6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -0.25, -0.1, -6, 4, 3, 2, 1, 0.5]) * s   # midpoints
    R = R.reshape(rows, D).astype(np.float32)
    for gscale in (float(np.abs(R).max() / (6 * 448)), 1.0, 1e-3):
        codes, scales = B.dllm_nvfp4_quantize(torch.from_numpy(R).cuda(), gscale)
        torch.cuda.synchronize()
        c_ref, s_ref = cl.nvfp4_quantize(R, gscale)
        np.testing.assert_array_equal(scales.cpu().numpy(), s_ref)
        np.testing.assert_array_equal(_unpack(codes), c_ref)
        # the round trip: dequantised values bit-exact (one fp32 rounding, by the tensor scale)
        deq = B.dllm_nvfp4_dequantize(codes, scales, gscale).cpu().numpy()
        want = cl.nvfp4_dequantize(c_ref, s_ref, gscale).astype(np.float32)
        np.testing.assert_array_equal(deq.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("kc", [0, 3, 16, 40])
def test_cluster_select_parity(B, kc):
    g = synth.rng(11 + kc)
    Bq, N, D, K = 2, 500, 128, 16
    Cp = g.standard_normal((Bq, K, D)).astype(np.float32)
    Cn = (Cp + g.uniform(0, 1, (Bq, K, 1)) * g.standard_normal((Bq, K, D))).astype(np.float32)
    Cn[0, 3] = 0.0                                                       # a zero centroid: drift 1
    a = g.integers(0, K, (Bq, N)).astype(np.int32)
    idx, cnt = B.dllm_cluster_select(torch.from_numpy(Cn).cuda(), torch.from_numpy(Cp).cuda(),
                                     torch.from_numpy(a).cuda(), kc)
    torch.cuda.synchronize()
    for b in range(Bq):
        d = np.sort(cl.cluster_drift(Cn[b], Cp[b]))[::-1]
        if 0 < kc < K:
            assert d[kc - 1] - d[kc] > 1e-5
        rows, _ = cl.select_clusters(Cn[b], Cp[b], a[b], kc)
        assert int(cnt[b]) == rows.size
        got = idx[b].cpu().numpy()
        np.testing.assert_array_equal(got[:rows.size], rows)
        assert np.all(got[rows.size:] == -1)
