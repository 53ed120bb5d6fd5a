"""Pins for the oracle's cluster-granular proxy (Polestar, "2. A. Polestar-Cache", local
window and clustering): spherical k-means against closed-form geometry, the E2M1 / E4M3
roundings against the formats' definitions (every code maps to itself, midpoints go to
the even code, saturation), NVFP4 exactness on a representable block and its error bound,
and the cluster selection against a hand example."""
import math

import numpy as np
import pytest

from oracle import cluster as cl
from sparse_kv_cache_rank_gb300 import synth


def _circle(deg):
    r = np.deg2rad(np.asarray(deg, dtype=np.float64))
    return np.stack([np.cos(r), np.sin(r)], axis=1)


def test_kmeans_two_arcs_closed_form():
    """Unit vectors at 0, 10 and 170, 180 degrees, centroids started at 45 and 135: the
    clusters are the two arcs and the centroids their bisectors (5 and 175 degrees)."""
    X = _circle([0, 10, 170, 180]) * np.array([[1.0], [2.0], [0.5], [3.0]])   # norms do not matter
    a, C = cl.spherical_kmeans(X, _circle([45, 135]), 5)
    np.testing.assert_array_equal(a, [0, 0, 1, 1])
    np.testing.assert_allclose(C, _circle([5, 175]), atol=1e-12)


def test_kmeans_single_cluster_is_mean_direction_and_scale_free():
    g = synth.rng(1)
    X = g.standard_normal((40, 6)) + np.array([3.0, 0, 0, 0, 0, 0])
    a, C = cl.spherical_kmeans(X, g.standard_normal((1, 6)), 3)
    U = X / np.linalg.norm(X, axis=1, keepdims=True)
    m = U.sum(0)
    np.testing.assert_allclose(C[0], m / np.linalg.norm(m), atol=1e-12)
    a2, C2 = cl.spherical_kmeans(X * g.uniform(0.1, 10, (40, 1)), g.standard_normal((1, 6)), 3)
    np.testing.assert_allclose(C2, C, atol=1e-12)


def test_kmeans_ties_and_empty_clusters():
    """Equal cosines go to the lower cluster; a cluster nobody joins keeps its centroid."""
    X = _circle([90, 90])
    a0, _ = cl.spherical_kmeans(X, _circle([0, 180, 300]), 0)
    np.testing.assert_array_equal(a0, [0, 0])      # cos 0 to both 0 and 180 degrees: the lower
    a, C = cl.spherical_kmeans(X, _circle([0, 180, 300]), 2)
    np.testing.assert_array_equal(a, [0, 0])
    np.testing.assert_allclose(C[1], _circle([180])[0], atol=1e-15)
    np.testing.assert_allclose(C[2], _circle([300])[0], atol=1e-15)


def test_residual_norm_identity():
    """|x - |x| c|^2 = 2 |x|^2 (1 - cos(x, c)) for a unit centroid c; 0 when x is along c."""
    g = synth.rng(2)
    X = g.standard_normal((20, 8))
    C = cl._unit_rows(g.standard_normal((3, 8)))
    a = g.integers(0, 3, 20)
    R = cl.residuals(X, C, a)
    n = np.linalg.norm(X, axis=1)
    cos = (X * C[a]).sum(1) / n
    np.testing.assert_allclose((R * R).sum(1), 2 * n * n * (1 - cos), rtol=1e-12)
    assert np.abs(cl.residuals(C * 3.0, C, np.arange(3))).max() < 1e-15


def test_e2m1_definition():
    grid = cl.E2M1_GRID
    for code, v in enumerate(grid):                      # every value maps to itself
        assert cl.e2m1_round(v)[1] == code and cl.e2m1_round(-v)[0] == -v
    mids = (grid[:-1] + grid[1:]) / 2
    _, c = cl.e2m1_round(mids)                           # midpoints -> the even code
    assert np.all(c % 2 == 0)
    assert cl.e2m1_round(100.0)[1] == 7 and cl.e2m1_round(-100.0)[1] == 15
    x = np.linspace(-7, 7, 2001)
    assert np.all(np.diff(cl.e2m1_round(x)[0]) >= 0)       # monotone
    assert cl.e2m1_round(-0.1)[1] == 8                   # sign kept on a zero result


def test_e4m3_definition():
    vals = cl.E4M3_VALUES
    assert vals[126] == 448.0 and vals[1] == 2.0 ** -9 and vals[8] == 2.0 ** -6
    assert np.all(np.diff(vals) > 0)
    for code in range(0, 127, 5):
        assert cl.e4m3_round(vals[code])[1] == code
    mids = (vals[:-1] + vals[1:]) / 2
    assert np.all(cl.e4m3_round(mids)[1] % 2 == 0)
    assert cl.e4m3_round(1e6)[1] == 126


def test_nvfp4_exact_on_representable_block_and_bound():
    """A block whose amax / 6 is a power of two and whose elements lie on the scaled grid
    comes back exactly; random data stays within the grid's half-spacing at the block
    scale (plus the scale's own rounding at the top of the range)."""
    s = 2.0 ** -3
    vals = np.array([6, -4, 3, 0.5, 0, -1.5, 2, 1, -6, 4, 0, 0.5, -0.5, 1.5, 3, -2]) * s
    codes, sc = cl.nvfp4_quantize(vals[None, :], 1.0)
    np.testing.assert_array_equal(cl.nvfp4_dequantize(codes, sc, 1.0)[0], vals)
    g = synth.rng(3)
    R = g.standard_normal((8, 64)).astype(np.float32) * 0.1
    gscale = float(np.abs(R).max() / (6 * 448))
    codes, sc = cl.nvfp4_quantize(R, gscale)
    Rh = cl.nvfp4_dequantize(codes, sc, gscale)
    blk = np.abs(R).reshape(8, 4, 16).max(-1)
    step = cl.E4M3_VALUES[sc] * np.float32(gscale)
    bound = np.maximum(step, blk / 8)[..., None].repeat(16, -1).reshape(8, 64)   # grid spacing <= 2 steps
    assert np.all(np.abs(R - Rh) <= bound + 1e-12)
    z_codes, z_sc = cl.nvfp4_quantize(np.zeros((2, 32)), 1.0)
    assert not z_codes.any() and not z_sc.any()


def test_cluster_selection_hand_example():
    C_prev = _circle([0, 90, 180, 270])
    C_now = _circle([30, 90, 200, 270])          # drifts: 1 - cos 30, 0, 1 - cos 20, 0
    a = np.array([0, 1, 2, 3, 0, 2, 1])
    rows, chosen = cl.select_clusters(C_now, C_prev, a, 1)
    np.testing.assert_array_equal(chosen, [0])
    np.testing.assert_array_equal(rows, [0, 4])
    rows, chosen = cl.select_clusters(C_now, C_prev, a, 3)    # tie at 0 between 1 and 3 -> 1
    np.testing.assert_array_equal(chosen, [0, 1, 2])
    np.testing.assert_array_equal(rows, [0, 1, 2, 4, 5, 6])
    assert cl.select_clusters(C_now, C_prev, a, 0)[0].size == 0
    d = cl.cluster_drift(C_now, C_prev)
    assert d[0] == pytest.approx(1 - math.cos(math.radians(30)))
