"""Pins for the oracle's layer refresh (SPA-Cache, "3. Sparse execution"): the
sparse Q/K/V at the selected rows, attention of those queries over the partially
updated cache, FFN on the sparse attention output, and an output written only at
the selected rows.  Structured weights reduce the layer to closed forms that a
transposed operand, a wrong head mapping, a wrong softmax scale, a wrong rotary
pairing or a missing residual would break."""
import math

import numpy as np
import pytest

from sparse_kv_cache_rank_gb300 import synth


def _zeros(d, n_q, n_kv, hd, F):
    return {
        "w_q": np.zeros((n_q * hd, d), np.float32), "w_k": np.zeros((n_kv * hd, d), np.float32),
        "w_v": np.zeros((n_kv * hd, d), np.float32), "w_o": np.zeros((d, n_q * hd), np.float32),
        "w_g": np.zeros((F, d), np.float32), "w_u": np.zeros((F, d), np.float32),
        "w_d": np.zeros((d, F), np.float32),
        "gamma1": np.ones(d, np.float32), "gamma2": np.ones(d, np.float32),
    }


def _perm_matrix(perm):
    n = len(perm)
    M = np.zeros((n, n), np.float32)
    M[np.arange(n), perm] = 1.0            # (x M^T)[j] = x[perm[j]]
    return M


def _rms(x, gamma, eps):
    x = x.astype(np.float64)
    return x / np.sqrt((x * x).mean(-1, keepdims=True) + eps) * gamma


def _all_rows(B, N):
    idx = np.tile(np.arange(N, dtype=np.int32), (B, 1))
    return idx, np.full(B, N, np.int32)


def test_uniform_attention_with_permutation_weights(orc):
    """W_q = W_k = 0 -> every score is 0 -> attention is the mean of V.
    W_V and W_O are permutations that are not involutions, so a transposed
    weight would pick different coordinates."""
    d, n_q, n_kv, hd, F, N = 8, 2, 2, 4, 4, 7
    pv = np.array([3, 0, 5, 1, 7, 2, 4, 6])
    po = np.array([1, 2, 3, 4, 5, 6, 7, 0])
    w = _zeros(d, n_q, n_kv, hd, F)
    w["w_v"] = _perm_matrix(pv)
    w["w_o"] = _perm_matrix(po)
    w["gamma1"] = (0.5 + synth.rng(1).random(d)).astype(np.float32)
    L = orc.Layer(w, n_q, n_kv, hd, eps=1e-5)
    H = synth.rng(2).standard_normal((1, N, d)).astype(np.float32)
    K, V, O = orc.layer_full(L, H)
    xn = _rms(H[0], w["gamma1"], 1e-5)
    v = xn[:, pv]
    a = v.mean(0)
    want = H[0] + a[po][None, :]
    np.testing.assert_allclose(V[0], v, rtol=1e-6, atol=1e-7)
    assert (K == 0).all()
    np.testing.assert_allclose(O[0], want, rtol=1e-6, atol=1e-6)


def test_softmax_scale_two_keys(orc):
    """Two orthogonal keys and a query along the first: the weight on key 0 is the
    logistic of the score gap, with scores scaled by 1/sqrt(hd)."""
    d = hd = 4
    alpha = 0.7
    w = _zeros(d, 1, 1, hd, 2)
    w["w_q"] = (alpha * np.eye(d)).astype(np.float32)
    w["w_k"] = np.eye(d, dtype=np.float32)
    w["w_v"] = np.eye(d, dtype=np.float32)
    w["w_o"] = np.eye(d, dtype=np.float32)
    L = orc.Layer(w, 1, 1, hd, eps=0.0, use_rope=False)
    H = np.zeros((1, 2, d), np.float32)
    H[0, 0, 0] = 2.0          # mean square 1 -> RMSNorm leaves it unchanged
    H[0, 1, 1] = 2.0
    _, _, O = orc.layer_full(L, H)
    gap = (2 * alpha * 2) / math.sqrt(hd)          # <q, k0> - <q, k1> = 4 alpha, / sqrt(hd)
    p0 = 1.0 / (1.0 + math.exp(-gap))
    want0 = np.array([2 + 2 * p0, 2 * (1 - p0), 0, 0])
    np.testing.assert_allclose(O[0, 0], want0, rtol=1e-6)


def test_gqa_head_mapping(orc):
    """n_q = 4, n_kv = 2: query heads 0,1 read KV head 0 and heads 2,3 read KV head 1."""
    d, n_q, n_kv, hd, N = 8, 4, 2, 2, 5
    w = _zeros(d, n_q, n_kv, hd, 2)
    w["w_v"] = np.eye(n_kv * hd, d, dtype=np.float32)        # v = xn[0:4]
    w["w_o"] = np.eye(d, dtype=np.float32)
    L = orc.Layer(w, n_q, n_kv, hd, eps=1e-5)
    H = synth.rng(3).standard_normal((1, N, d)).astype(np.float32)
    _, _, O = orc.layer_full(L, H)
    xn = _rms(H[0], w["gamma1"], 1e-5)
    m = xn[:, :4].mean(0)
    a = np.concatenate([m[0:2], m[0:2], m[2:4], m[2:4]])
    np.testing.assert_allclose(O[0] - H[0], np.broadcast_to(a, (N, d)), rtol=1e-6, atol=1e-6)


def test_swiglu_ffn_closed_form(orc):
    """Zero attention path; W_g = c I, W_u = I, W_d = I: out = h + SiLU(c xn2) * xn2."""
    d, N, c = 6, 4, 1.3
    w = _zeros(d, 1, 1, d, d)
    w["w_g"] = (c * np.eye(d)).astype(np.float32)
    w["w_u"] = np.eye(d, dtype=np.float32)
    w["w_d"] = np.eye(d, dtype=np.float32)
    w["gamma2"] = (0.5 + synth.rng(4).random(d)).astype(np.float32)
    L = orc.Layer(w, 1, 1, d, eps=1e-5)
    H = synth.rng(5).standard_normal((1, N, d)).astype(np.float32)
    H[0, 2] = 0.0                                   # SiLU(0) = 0: row stays 0
    _, _, O = orc.layer_full(L, H)
    xn2 = _rms(H[0], w["gamma2"], 1e-5)
    g = c * xn2
    want = H[0] + g / (1.0 + np.exp(-g)) * xn2
    np.testing.assert_allclose(O[0], want, rtol=1e-6, atol=1e-7)
    assert (O[0, 2] == 0).all()


def test_rope_closed_form(orc):
    """Rotate-half pairs (i, i + hd/2) turn by pos * theta^(-2i/hd)."""
    e = np.eye(4, dtype=np.float32)
    out = orc.rope_row(e[1], 100)                   # pair (1,3), freq 1e4^-0.5 = 0.01
    np.testing.assert_allclose(out, [0, math.cos(1.0), 0, math.sin(1.0)], atol=1e-7)
    out = orc.rope_row(e[0], 3)                     # pair (0,2), freq 1
    np.testing.assert_allclose(out, [math.cos(3.0), 0, math.sin(3.0), 0], atol=1e-7)
    out = orc.rope_row(e[2], 3)
    np.testing.assert_allclose(out, [-math.sin(3.0), 0, math.cos(3.0), 0], atol=1e-7)
    x = synth.rng(6).standard_normal(64).astype(np.float32)
    y = orc.rope_row(orc.rope_row(x, 17), 25)
    np.testing.assert_allclose(y, orc.rope_row(x, 42), rtol=1e-5, atol=1e-5)
    assert math.isclose(np.linalg.norm(orc.rope_row(x, 999)), np.linalg.norm(x), rel_tol=1e-6)


def test_refresh_rotates_keys_at_their_own_position(orc):
    """All rows equal: the key written for row i is the row-0 key rotated to position i,
    also when only rows {2, 5} are refreshed (position = row index, not slot)."""
    d, hd, N = 16, 16, 8
    w = synth.layer_weights(synth.LayerShape("t", 1, N, d, 1, 1, hd, 8, 4, 0.5, "f32"), 7)
    L = orc.Layer(w, 1, 1, hd)
    row = synth.rng(8).standard_normal(d).astype(np.float32)
    H = np.tile(row, (1, N, 1)).astype(np.float32)
    K, V, O = orc.layer_full(L, H)
    for i in range(N):
        np.testing.assert_allclose(K[0, i], orc.rope_row(K[0, 0], i), rtol=1e-5, atol=1e-6)
    K2 = np.zeros_like(K)
    V2 = np.zeros_like(V)
    O2 = np.zeros_like(O)
    idx = np.array([[2, 5] + [-1] * (N - 2)], np.int32)
    orc.layer_refresh(L, H, idx, np.array([2], np.int32), K2, V2, O2)
    np.testing.assert_allclose(K2[0, 5], orc.rope_row(K[0, 0], 5), rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(K2[0, 2], K[0, 2], rtol=0, atol=0)


def test_attention_rows_properties(orc):
    """Softmax weights sum to one (V all ones -> output ones); equal keys -> mean of V."""
    n_q, n_kv, hd, N = 4, 2, 8, 9
    d = n_q * hd
    L = orc.Layer(_zeros(d, n_q, n_kv, hd, 2), n_q, n_kv, hd)
    g = synth.rng(9)
    Q = g.standard_normal((3, n_q * hd)).astype(np.float32)
    K = g.standard_normal((N, n_kv * hd)).astype(np.float32)
    A = orc.attention_rows(L, Q, K, np.ones((N, n_kv * hd), np.float32))
    np.testing.assert_allclose(A, 1.0, rtol=1e-6)
    Keq = np.tile(K[:1], (N, 1))
    Vr = g.standard_normal((N, n_kv * hd)).astype(np.float32)
    A = orc.attention_rows(L, Q, Keq, Vr)
    m = Vr.astype(np.float64).mean(0)
    want = np.concatenate([m[0:hd], m[0:hd], m[hd:], m[hd:]])
    np.testing.assert_allclose(A, np.broadcast_to(want, A.shape), rtol=1e-5, atol=1e-6)


def _small():
    sh = synth.LayerShape("small", B=2, N=24, d=64, n_q=4, n_kv=2, hd=16, F=96, r=8,
                          rho=0.25, dtype="f32")
    return sh, synth.layer_weights(sh, 11, std=0.1)


def test_full_selection_equals_full_forward(orc):
    """Invariant: refreshing every row is the full recomputation."""
    sh, w = _small()
    L = orc.Layer(w, sh.n_q, sh.n_kv, sh.hd)
    Hp, Hc, _ = synth.hidden_pair(sh, 12)
    K, V, O = orc.layer_full(L, Hp)                        # stale caches
    Kf, Vf, Of = orc.layer_full(L, Hc)                     # reference
    idx, cnt = _all_rows(sh.B, sh.N)
    orc.layer_refresh(L, Hc, idx, cnt, K, V, O)
    np.testing.assert_allclose(K, Kf, rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(V, Vf, rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(O, Of, rtol=1e-6, atol=1e-6)


def test_unselected_rows_untouched_and_consistent_cache_reproduced(orc):
    sh, w = _small()
    L = orc.Layer(w, sh.n_q, sh.n_kv, sh.hd)
    Hp, Hc, _ = synth.hidden_pair(sh, 13)
    K, V, O = orc.layer_full(L, Hp)
    idx = np.full((sh.B, sh.N), -1, np.int32)
    sel = [np.array([0, 5, 6, 23]), np.array([1, 2, 17])]
    for b, s in enumerate(sel):
        idx[b, :len(s)] = s
    cnt = np.array([len(s) for s in sel], np.int32)
    # (iii) same input as the cache was built from -> refreshed rows reproduce the cache
    K1, V1, O1 = K.copy(), V.copy(), O.copy()
    orc.layer_refresh(L, Hp, idx, cnt, K1, V1, O1)
    np.testing.assert_allclose(O1, O, rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(K1, K, rtol=1e-6, atol=1e-7)
    # (ii) new input -> only the selected rows change, the rest stay bitwise equal
    pc = np.zeros((sh.B, sh.N, sh.r), np.float32)
    cur = np.ones((sh.B, sh.N, sh.r), np.float32)
    K2, V2, O2 = K.copy(), V.copy(), O.copy()
    orc.layer_refresh(L, Hc, idx, cnt, K2, V2, O2, proxy_cache=pc, proxy_cur=cur)
    for b, s in enumerate(sel):
        keep = np.setdiff1d(np.arange(sh.N), s)
        assert (K2[b, keep] == K[b, keep]).all() and (V2[b, keep] == V[b, keep]).all()
        assert (O2[b, keep] == O[b, keep]).all()
        assert not np.allclose(O2[b, s], O[b, s])
        assert (pc[b, s] == 1).all() and (pc[b, keep] == 0).all()


def test_sampled_outputs_match_full_refresh(orc):
    sh, w = _small()
    L = orc.Layer(w, sh.n_q, sh.n_kv, sh.hd)
    Hp, Hc, _ = synth.hidden_pair(sh, 14)
    K, V, O = orc.layer_full(L, Hp)
    idx, cnt = _all_rows(sh.B, sh.N)
    full = [a.copy() for a in (K, V, O)]
    orc.layer_refresh(L, Hc, idx, cnt, *full)
    mask = np.zeros((sh.B, sh.N), np.uint8)
    mask[:, ::5] = 1
    part = [a.copy() for a in (K, V, O)]
    orc.layer_refresh(L, Hc, idx, cnt, *part, out_mask=mask)
    m = mask.astype(bool)
    np.testing.assert_array_equal(part[2][m], full[2][m])
    np.testing.assert_array_equal(part[0], full[0])
