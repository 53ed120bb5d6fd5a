"""GPU-vs-oracle parity through the C ABI (via the thin torch binding).

Both sides start from the same seeded inputs and each decides on its own values (the
oracle never receives a value the GPU computed).  Sets and tokens: equal, except
decisions inside the 1e-5 near-tie band of the oracle's own scores.  fp32 reductions: 1e-4 relative.  Layer outputs:
bf16 max-relative error <= 2e-2 with cosine >= 0.999; fp32 <= 1e-4.
"""
import dataclasses

import numpy as np
import pytest

from sparse_kv_cache_rank_gb300 import synth
from cases import (assert_close_layer, assert_drift_close, assert_update_close, forced_rows, layer_case,
                   match_selection, normwise_rel, to_dev, to_np, torch_dtype, FP32_REDUCTION_RTOL, TIE_BAND)

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


# shapes: several tiles and ragged tails on every axis the kernels tile
SMALL_BF16 = synth.LayerShape("small-bf16-gqa", B=2, N=200, d=256, n_q=4, n_kv=2, hd=64, F=320,
                              r=64, rho=0.25, dtype="bf16", prompt=100, k_recent=4)
MID_BF16 = synth.LayerShape("mid-bf16-hd128", B=1, N=333, d=512, n_q=4, n_kv=4, hd=128, F=704,
                            r=128, rho=0.3, dtype="bf16", prompt=200)
TINY_BF16 = dataclasses.replace(synth.TINY, name="tiny-bf16", dtype="bf16")
# fp32 on the CUDA cores with 128-dim heads, GQA and a ragged key tail per attention warp
MID_F32_GQA = synth.LayerShape("mid-f32-hd128-gqa", B=2, N=301, d=512, n_q=4, n_kv=2, hd=128, F=640,
                               r=32, rho=0.2, dtype="f32", prompt=200)


# --------------------------------------------------------------------------- proxy
@pytest.mark.parametrize("shape", [synth.TINY, TINY_BF16, SMALL_BF16, MID_BF16], ids=lambda s: s.name)
def test_proxy_score_parity(B, orc, shape):
    c = layer_case(orc, shape, 10)
    dt = torch_dtype(shape)
    cur, drift = B.dllm_proxy_score(to_dev(c.H_cur, dt), to_dev(c.P.T.copy(), dt), to_dev(c.pc0))
    torch.cuda.synchronize()
    cur_o, drift_o = orc.proxy_score(c.H_cur, c.P, c.pc0)
    assert normwise_rel(to_np(cur), cur_o) < FP32_REDUCTION_RTOL
    assert_drift_close(to_np(drift), drift_o)


def test_proxy_identical_inputs_zero_drift(B, orc):
    c = layer_case(orc, SMALL_BF16, 11)
    H = to_dev(c.H_prev, torch.bfloat16)
    Pt = to_dev(c.P.T.copy(), torch.bfloat16)
    cur, _ = B.dllm_proxy_score(H, Pt, torch.ones((2, 200, 64), device="cuda"))
    _, drift = B.dllm_proxy_score(H, Pt, cur.clone())
    assert (drift == 0).all().item()


@pytest.mark.parametrize("N", [1024, 4096])
def test_proxy_llada_width(B, orc, N):
    """LLaDA-8B width (d = 4096, r = 128) over N rows; oracle on every row."""
    g = synth.rng(12)
    d, r = 4096, 128
    H0 = synth.round_bf16(g.standard_normal((1, N, d), dtype=np.float32))
    H1 = synth.round_bf16(H0 + g.standard_normal((1, N, d), dtype=np.float32) * np.float32(0.05))
    P = synth.round_bf16((g.standard_normal((d, r)) * 0.02).astype(np.float32))
    pc, _ = orc.proxy_score(H0, P, np.ones((1, N, r), np.float32))
    cur, drift = B.dllm_proxy_score(to_dev(H1, torch.bfloat16), to_dev(P.T.copy(), torch.bfloat16),
                                    to_dev(pc))
    cur_o, drift_o = orc.proxy_score(H1, P, pc)
    assert normwise_rel(to_np(cur), cur_o) < FP32_REDUCTION_RTOL
    assert_drift_close(to_np(drift), drift_o)


@pytest.mark.parametrize("Bq,N,d,r", [
    (1, 1024, 4096, 128),   # 8 independent K slices summed by the cosine kernel
    (10, 4096, 128, 128),   # 320 token tiles of 128 rows fill the GPU: drift in the epilogue
    (10, 3950, 256, 96),    # the same with a ragged last tile and a proxy narrower than the
                            # tile (the fourth TMEM lane quarter holds no feature)
    (2, 9, 128, 64),        # d = 128 too short to split: one ragged tile, drift in the epilogue
    (3, 17, 256, 32),       # one ragged tile in 2 K slices, cosine kernel
    (1, 300, 512, 256),     # r > 128: K slices and the cosine kernel
], ids=["slices8", "epilogue-40960rows", "epilogue-r96-ragged", "epilogue-short-k", "slices2-r32",
        "slices-r256"])
def test_proxy_plans_parity(B, orc, Bq, N, d, r):
    """Every launch plan of the singular proxy and its drift (SPA-Cache, "1. Update
    identification via singular proxy") against the oracle on every row, with the
    degenerate rows of the drift's definition: a zero current proxy (drift 1), a zero
    cached proxy (drift 1) and both zero (drift 0); a second call against the first
    call's own proxies gives exactly zero drift on every row."""
    g = synth.rng(14 + N + r)
    H0 = synth.round_bf16(g.standard_normal((Bq, N, d), dtype=np.float32))
    H1 = synth.round_bf16(H0 + g.standard_normal((Bq, N, d), dtype=np.float32) * np.float32(0.05))
    P = synth.round_bf16((g.standard_normal((d, r)) * 0.02).astype(np.float32))
    pc, _ = orc.proxy_score(H0, P, np.ones((Bq, N, r), np.float32))
    last = Bq - 1
    H1[0, 1] = 0.0                  # current proxy zero, cached not: drift 1
    pc[last, N - 1] = 0.0           # cached proxy zero, current not: drift 1
    if N > 3:
        H1[0, 3] = 0.0              # both zero: drift 0
        pc[0, 3] = 0.0
    Hd = to_dev(H1, torch.bfloat16)
    Pt = to_dev(P.T.copy(), torch.bfloat16)
    cur, drift = B.dllm_proxy_score(Hd, Pt, to_dev(pc))
    torch.cuda.synchronize()
    cur_o, drift_o = orc.proxy_score(H1, P, pc)
    assert normwise_rel(to_np(cur), cur_o) < FP32_REDUCTION_RTOL
    dg = to_np(drift)
    assert_drift_close(dg, drift_o)
    assert dg[0, 1] == 1.0 and dg[last, N - 1] == 1.0
    if N > 3:
        assert dg[0, 3] == 0.0
    _, again = B.dllm_proxy_score(Hd, Pt, cur.clone())
    assert (again == 0).all().item()


# --------------------------------------------------------------------------- selection
@pytest.mark.parametrize("Bq,N,k,F,ties", [(1, 1, 1, 0, False), (3, 37, 5, 3, True),
                                            (2, 1024, 164, 0, False), (1, 1024, 164, 40, True),
                                            (4, 5000, 800, 17, True), (1, 16384, 2000, 64, False),
                                            (2, 300, 0, 8, False), (2, 300, 400, 8, False)])
def test_select_bit_exact(B, orc, Bq, N, k, F, ties):
    g = synth.rng(1000 + N + k)
    if ties:
        drift = g.choice(np.array([0, 1e-7, 1e-3, 2e-3, 0.1, 0.1, 0.5], np.float32), size=(Bq, N))
    else:
        drift = (g.random((Bq, N)) ** 3).astype(np.float32)
    forced = g.integers(-3, N + 3, size=(Bq, F)).astype(np.int32) if F else None
    idx, cnt = B.dllm_select_topk(to_dev(drift), to_dev(forced) if F else None, k)
    idx_o, cnt_o = orc.select_topk(drift, forced, k)
    np.testing.assert_array_equal(to_np(cnt), cnt_o)
    np.testing.assert_array_equal(to_np(idx), idx_o)


def test_select_degenerate(B, orc):
    z = np.zeros((2, 64), np.float32)
    idx, cnt = B.dllm_select_topk(to_dev(z), None, 10)
    assert (to_np(cnt) == 0).all() and (to_np(idx) == -1).all()
    nan = np.full((1, 64), np.nan, np.float32)
    nan[0, 9] = 0.3
    idx, cnt = B.dllm_select_topk(to_dev(nan), None, 10)
    assert to_np(cnt)[0] == 1 and to_np(idx)[0, 0] == 9


# --------------------------------------------------------------------------- refresh
def _step(B, orc, c, k, forced, sample=None, sample_seed=0, one_call=False):
    """One step on the GPU and on the oracle, each from the same seeded inputs and each
    deciding on its own values: the oracle scores, selects and refreshes by itself.
    sample=n: the oracle computes the layer outputs of n rows drawn from its own
    selection per sequence (large shapes); K/V of every selected row are always computed."""
    sh = c.shape
    dt = torch_dtype(sh)
    Bn, N = sh.B, sh.N
    H = to_dev(c.H_cur, dt)
    pc = to_dev(c.pc0)
    Pt = to_dev(c.P.T.copy(), dt)
    fo = to_dev(forced) if forced is not None else None
    k_max = min(N, k + (0 if forced is None else forced.shape[1]))
    layer = B.dllm_pack_layer({n: to_dev(v, dt) for n, v in c.w.items()}, sh.n_q, sh.n_kv, sh.hd,
                              eps=sh.eps, rope_theta=sh.rope_theta)
    K = to_dev(c.K0, dt)
    V = to_dev(c.V0, dt)
    O = to_dev(c.O0, dt)
    if one_call:   # proxy, selection and refresh through dllm_layer_step
        cur = torch.empty((Bn, N, sh.r), dtype=torch.float32, device="cuda")
        drift = torch.empty((Bn, N), dtype=torch.float32, device="cuda")
        idx = torch.empty((Bn, N), dtype=torch.int32, device="cuda")
        cnt = torch.empty((Bn,), dtype=torch.int32, device="cuda")
        B.dllm_layer_step(layer, Pt, H, pc, cur, drift, fo, k, idx, cnt, K, V, O)
    else:
        cur, drift = B.dllm_proxy_score(H, Pt, pc)
        idx, cnt = B.dllm_select_topk(drift, fo, k)
        B.dllm_sparse_layer_refresh(layer, H, idx, cnt, k_max, K, V, O, pc, cur)
    torch.cuda.synchronize()
    assert B.check_status() == 0
    g = dict(cur=to_np(cur), drift=to_np(drift), idx=to_np(idx), cnt=to_np(cnt), K=to_np(K),
             V=to_np(V), O=to_np(O), pc=to_np(pc))
    cur_o, drift_o = orc.proxy_score(c.H_cur, c.P, c.pc0)
    idx_o, cnt_o = orc.select_topk(drift_o, forced, k)
    out_mask = None
    if sample is not None:
        out_mask = np.zeros((Bn, N), np.uint8)
        for b in range(Bn):
            I = idx_o[b, :cnt_o[b]]
            out_mask[b, I[synth.rng(sample_seed + b).permutation(len(I))[:sample]]] = 1
    L = orc.Layer(c.w, sh.n_q, sh.n_kv, sh.hd, eps=sh.eps, rope_theta=sh.rope_theta)
    Ko, Vo, Oo, pco = c.K0.copy(), c.V0.copy(), c.O0.copy(), c.pc0.copy()
    orc.layer_refresh(L, c.H_cur, idx_o, cnt_o, Ko, Vo, Oo, pco, cur_o, out_mask=out_mask)
    o = dict(cur=cur_o, drift=drift_o, idx=idx_o, cnt=cnt_o, K=Ko, V=Vo, O=Oo, pc=pco, mask=out_mask)
    return g, o


def _compare_step(c, g, o, forced, k):
    sh = c.shape
    assert_drift_close(g["drift"], o["drift"])
    sets = match_selection(g["idx"], g["cnt"], o["drift"], o["idx"], o["cnt"], forced, k)
    for b in range(sh.B):
        I = g["idx"][b, :g["cnt"][b]]
        common = sets[b][0]
        rest = np.setdiff1d(np.arange(sh.N), I)
        # untouched rows keep their exact bits; the refreshed rows' cached proxies are this step's
        for name, ref in (("K", c.K0), ("V", c.V0), ("O", c.O0), ("pc", c.pc0)):
            np.testing.assert_array_equal(g[name][b, rest], ref[b, rest], err_msg=name)
        np.testing.assert_array_equal(g["pc"][b, I], g["cur"][b, I])
        assert normwise_rel(g["pc"][b, common], o["pc"][b, common]) < FP32_REDUCTION_RTOL
        assert_close_layer(g["K"][b, common], o["K"][b, common], sh.dtype, f"K b={b}")
        assert_close_layer(g["V"][b, common], o["V"][b, common], sh.dtype, f"V b={b}")
        rows = common if o["mask"] is None else common[o["mask"][b, common] != 0]
        assert len(rows) > 0
        assert_close_layer(g["O"][b, rows], o["O"][b, rows], sh.dtype, f"H_out b={b}")
        # the update itself (output minus input), not only the residual stream
        assert_update_close(g["O"][b, rows], o["O"][b, rows], c.H_cur[b, rows], sh.dtype,
                            f"H_out - H_in b={b}")


@pytest.mark.parametrize("one_call", [False, True], ids=["three-calls", "layer-step"])
@pytest.mark.parametrize("shape", [synth.TINY, TINY_BF16, SMALL_BF16, MID_BF16, MID_F32_GQA], ids=lambda s: s.name)
def test_refresh_step_parity(B, orc, shape, one_call):
    c = layer_case(orc, shape, 20)
    forced = forced_rows(shape, 21) if shape.k_recent else None
    k = orc.budget(shape.rho, shape.N)
    g, o = _step(B, orc, c, k, forced, one_call=one_call)
    _compare_step(c, g, o, forced, k)


LONG_SMALL = synth.LayerShape("long-small-bf16", B=2, N=5000, d=128, n_q=2, n_kv=1, hd=64, F=128, r=32,
                              rho=0.02, dtype="bf16", prompt=4900, k_recent=4)


# 320 short sequences: the fused drift + selection grid (one CTA per sequence) would not
# fit the GPU at once, so the layer step falls back to the cosine kernel
MANY_SEQ = synth.LayerShape("many-seq-bf16", B=320, N=40, d=256, n_q=2, n_kv=1, hd=64, F=128, r=32,
                            rho=0.05, dtype="bf16", prompt=8, k_recent=2)


@pytest.mark.parametrize("shape", [SMALL_BF16, synth.TINY, LONG_SMALL, MANY_SEQ], ids=lambda s: s.name)
def test_layer_step_equals_three_calls(B, orc, shape):
    """dllm_layer_step (selection fused with the gather up to N = 4096 and, with K-slice
    partials, the drift computed by that kernel; the separate kernels beyond N = 4096 or
    when the fused grid would not fit the GPU at once) writes exactly what
    dllm_proxy_score, dllm_select_topk and dllm_sparse_layer_refresh write in sequence:
    the same arithmetic, bit for bit."""
    c = layer_case(orc, shape, 25, consistent=shape.N <= 1024)
    forced = forced_rows(shape, 26)
    k = orc.budget(shape.rho, shape.N)
    dt = torch_dtype(shape)
    layer = B.dllm_pack_layer({n: to_dev(v, dt) for n, v in c.w.items()}, shape.n_q, shape.n_kv, shape.hd,
                              eps=shape.eps, rope_theta=shape.rope_theta)
    outs = []
    for one in (False, True):
        H, Pt, pc = to_dev(c.H_cur, dt), to_dev(c.P.T.copy(), dt), to_dev(c.pc0)
        K, V, O = to_dev(c.K0, dt), to_dev(c.V0, dt), to_dev(c.O0, dt)
        fo = to_dev(forced)
        if one:
            cur = torch.empty((shape.B, shape.N, shape.r), device="cuda")
            drift = torch.empty((shape.B, shape.N), device="cuda")
            idx = torch.empty((shape.B, shape.N), dtype=torch.int32, device="cuda")
            cnt = torch.empty((shape.B,), dtype=torch.int32, device="cuda")
            B.dllm_layer_step(layer, Pt, H, pc, cur, drift, fo, k, idx, cnt, K, V, O)
        else:
            cur, drift = B.dllm_proxy_score(H, Pt, pc)
            idx, cnt = B.dllm_select_topk(drift, fo, k)
            B.dllm_sparse_layer_refresh(layer, H, idx, cnt, min(shape.N, k + forced.shape[1]), K, V, O, pc, cur)
        torch.cuda.synchronize()
        outs.append([t.clone() for t in (cur, drift, idx, cnt, K, V, O, pc)])
    assert B.check_status() == 0
    for name, a, b in zip(("cur", "drift", "idx", "count", "K", "V", "H_out", "proxy_cache"), *outs):
        assert torch.equal(a, b), name


@pytest.mark.parametrize("shape", [synth.TINY, SMALL_BF16], ids=lambda s: s.name)
def test_full_selection_is_full_recompute(B, orc, shape):
    """Selecting every row from stale caches equals the oracle's dense forward on H_t."""
    c = layer_case(orc, shape, 30)
    g, _ = _step(B, orc, c, shape.N, None)
    assert (g["cnt"] == shape.N).all()
    L = orc.Layer(c.w, shape.n_q, shape.n_kv, shape.hd, eps=shape.eps, rope_theta=shape.rope_theta)
    Kf, Vf, Of = orc.layer_full(L, c.H_cur)
    assert_close_layer(g["K"], Kf, shape.dtype, "K")
    assert_close_layer(g["V"], Vf, shape.dtype, "V")
    assert_close_layer(g["O"], Of, shape.dtype, "H_out")


def test_refresh_llada_layer_sampled(B, orc):
    """LLaDA-8B-shaped layer at full size (N=1024, d=4096, 32x128, F=12288, 16%):
    drift of every row, K/V of every selected row, layer outputs of 12 rows sampled from
    the oracle's selection."""
    sh = synth.LLADA_LAYER
    c = layer_case(orc, sh, 40, consistent=False, svd_proxy=False)
    k = orc.budget(sh.rho, sh.N)
    assert k == 164
    g, o = _step(B, orc, c, k, None, sample=12, sample_seed=41, one_call=True)
    _compare_step(c, g, o, None, k)
    # every strongly perturbed row is in the selection
    assert set(c.hot[0].tolist()) <= set(g["idx"][0, :g["cnt"][0]].tolist())


# --------------------------------------------------------------------------- vocabulary
@pytest.mark.parametrize("Bq,M,V,scale", [(1, 24, 4096, 1.0), (1, 24, 4096, 10.0),
                                          (2, 32, 126464, 0.43), (8, 32, 152064, 0.43),
                                          (3, 5, 7, 1.0), (1, 1000, 64, 4.0)])
def test_commit_entropy_parity(B, orc, Bq, M, V, scale):
    logits = synth.commit_logits(Bq, M, V, 50 + M, std=3.0 * scale)
    valid = np.ones((Bq, M), np.uint8)
    valid[-1, ::3] = 0
    tok, conf, ent, E, full = B.dllm_commit_entropy(to_dev(logits), to_dev(valid))
    torch.cuda.synchronize()
    am_o, pm_o, H_o = orc.vocab_stats(logits)
    v = valid.astype(bool)
    conf, ent = to_np(conf), to_np(ent)
    np.testing.assert_allclose(conf[v], pm_o[v], rtol=FP32_REDUCTION_RTOL, atol=1e-9)
    np.testing.assert_allclose(ent[v], H_o[v], rtol=FP32_REDUCTION_RTOL, atol=1e-6)
    assert (conf[~v] == 0).all() and (ent[~v] == 0).all()
    # the decisions against the oracle's own statistics: the argmax is taken on the same
    # fp32 logits on both sides, so tokens agree wherever no confidence lies within the
    # near-tie band of the threshold and the fallback row is not a near-tie
    t_r, E_r, f_r = orc.commit_rule(am_o, pm_o, H_o, valid)
    tok, E, full = to_np(tok), to_np(E), to_np(full)
    for b in range(Bq):
        pv = np.where(v[b], pm_o[b], -1.0)
        near = bool((np.abs(pv - 0.9) < TIE_BAND).any())
        if not (pv >= 0.9).any():       # fallback: the single most confident valid row
            top = np.sort(pv)[::-1]
            near |= bool(len(top) > 1 and top[1] >= 0 and top[0] - top[1] < TIE_BAND)
        if near:
            continue
        np.testing.assert_array_equal(tok[b], t_r[b])
        np.testing.assert_allclose(E[b], E_r[b], rtol=FP32_REDUCTION_RTOL, atol=1e-6)
        if abs(E_r[b] - 2.0) > FP32_REDUCTION_RTOL * 2.0:
            assert full[b] == f_r[b]


def test_commit_no_valid_rows(B):
    logits = torch.zeros((2, 4, 16), device="cuda")
    valid = torch.zeros((2, 4), dtype=torch.uint8, device="cuda")
    tok, conf, ent, E, full = B.dllm_commit_entropy(logits, valid)
    assert (tok == -1).all().item() and (E == 0).all().item() and (full == 0).all().item()


# --------------------------------------------------------------------------- plain GEMM
@pytest.mark.parametrize("M,N_out,K,splits", [(1, 32, 64, 0), (37, 96, 192, 0), (164, 512, 1024, 1),
                                              (164, 512, 1024, 4), (300, 384, 640, 0),
                                              (513, 256, 2048, 8), (64, 4096, 4096, 0),
                                              (164, 384, 12288, 0), (256, 1024, 4096, 0),
                                              (200, 2080, 1024, 0), (16, 128, 256, 0),
                                              (96, 160 * 128 + 96, 256, 0),
                                              (257, 1024, 512, 0), (516, 8192, 512, 0),
                                              (642, 8192, 512, 0), (705, 8192, 512, 0),
                                              (775, 8192, 512, 0), (838, 8192, 512, 0),
                                              (901, 8192, 512, 0)])
def test_gemm_bf16_parity(B, orc, M, N_out, K, splits):
    """The engine under every projection: X W^T against the oracle's double-precision
    projection (the proxy score computes exactly H . P), ragged M, K splits 1..8, long K
    over few weight tiles (automatic cluster split), a ragged last weight tile (2080 rows),
    tiny grids, and more weight tiles than SMs.  The last six have more than 256 tokens and
    8192 outputs, so that the planner's token-tile width is 160, 176, 192, 208, 224 and 256
    in turn, each with a ragged last token tile; (257, 1024, 512) gives no width enough
    tiles and takes the K split."""
    g = synth.rng(3000 + M + K)
    X = synth.round_bf16(g.standard_normal((M, K), dtype=np.float32))
    W = synth.round_bf16((g.standard_normal((N_out, K)) * 0.05).astype(np.float32))
    out = B.dllm_gemm_bf16(to_dev(X, torch.bfloat16), to_dev(W, torch.bfloat16), splits=splits)
    ref, _ = orc.proxy_score(X[None], np.ascontiguousarray(W.T), np.ones((1, M, N_out), np.float32))
    assert normwise_rel(to_np(out), ref[0]) < FP32_REDUCTION_RTOL


def _sampled_layer_parity(B, orc, sh, seed, n_sample=8):
    c = layer_case(orc, sh, seed, consistent=False, svd_proxy=False)
    k = orc.budget(sh.rho, sh.N)
    g, o = _step(B, orc, c, k, None, sample=n_sample, sample_seed=seed)
    _compare_step(c, g, o, None, k)
    for b in range(sh.B):
        hot, sel = set(c.hot[b].tolist()), set(g["idx"][b, :g["cnt"][b]].tolist())
        # the strongly perturbed rows come first: all of them when they fit the budget,
        # otherwise the budget is spent on them alone
        assert hot <= sel if len(hot) <= k else sel <= hot


def test_refresh_dream_layer_sampled(B, orc):
    """Dream-7B-shaped (Qwen2.5-7B layout) layer: d=3584, 28 query / 4 KV heads x 128
    (GQA group 7), F=18944, r=128, 16% of N=2048 -> k=328 per sequence; batch 2
    (the configuration's batch 8 changes only the number of independent sequences)."""
    sh = dataclasses.replace(synth.DREAM_STACK, name="dream7b-layer-b2", B=2, layers=1, V=0)
    _sampled_layer_parity(B, orc, sh, 70)


def test_refresh_long_context_point(B, orc):
    """Long-context sweep point: LLaDA-8B-shaped layer at N=8192 with a 5% update ratio."""
    sh = dataclasses.replace(synth.LLADA_LAYER, name="llada8b-N8192-rho0.05", N=8192, rho=0.05,
                             prompt=4096)
    _sampled_layer_parity(B, orc, sh, 71, n_sample=6)


def test_refresh_long_context_n2048_sixteenth(B, orc):
    """Long-context sweep point just past the few-token regime: LLaDA-8B-shaped layer at
    N = 2048 with 16 % (328 rows): the O and down projections (32 weight tiles x 3 token
    tiles of 128) run with a 3-way cluster K split so that every SM streams."""
    sh = dataclasses.replace(synth.LLADA_LAYER, name="llada8b-N2048-rho0.16", N=2048, rho=0.16, prompt=1024)
    p = B.dllm_gemm_plan(orc.budget(sh.rho, sh.N), sh.d, sh.d_q, sms=152)
    assert p["splits"] == 3 and p["tok_tiles"] == 3
    _sampled_layer_parity(B, orc, sh, 73, n_sample=6)


def test_refresh_long_context_batch4_half(B, orc):
    """Long-context sweep point with a batch and half the rows refreshed: LLaDA-8B-shaped
    layer at N = 2048, batch 4, 50 % (1024 rows per sequence, 4096 in all, the
    tensor-bound side of the sweep, taken by the one-call layer step); K/V of every
    selected row, outputs of 4 rows per sequence."""
    sh = dataclasses.replace(synth.LLADA_LAYER, name="llada8b-N2048-B4-rho0.5", N=2048, B=4, rho=0.5,
                             prompt=1024)
    c = layer_case(orc, sh, 72, consistent=False, svd_proxy=False)
    k = orc.budget(sh.rho, sh.N)
    assert k == 1024
    g, o = _step(B, orc, c, k, None, sample=4, sample_seed=72, one_call=True)
    _compare_step(c, g, o, None, k)


# --------------------------------------------------------------------------- attention alone
@pytest.mark.parametrize("Bq,N,k_max,n_q,n_kv,hd,live,growth", [
    (1, 1024, 164, 32, 32, 128, 164, 0), (2, 333, 150, 4, 2, 64, 150, 0), (1, 2048, 328, 28, 4, 128, 300, 0),
    # 64-dim heads over 16 key tiles per CTA (two softmax threads per row, pipelined)
    (4, 2048, 256, 16, 8, 64, 250, 0),
    # scores growing from key tile to key tile: every tile raises the rows' running
    # maximum (the streaming softmax rescales O at every tile), 128- and 64-dim heads
    (1, 2048, 328, 28, 4, 128, 300, 3), (4, 2048, 256, 16, 8, 64, 250, 3),
    (3, 200, 37, 8, 8, 128, 37, 0), (1, 129, 129, 2, 1, 64, 100, 0),
    # one key slice per CTA (the grid alone fills the GPU), a ragged second query tile
    (8, 256, 200, 28, 4, 128, 200, 0), (16, 150, 140, 16, 16, 64, 140, 0)])
def test_attention_parity(B, orc, Bq, N, k_max, n_q, n_kv, hd, live, growth):
    """Selected queries over the whole cache, non-causal, GQA, ragged key tiles and
    partially live query tiles, key slices merged in a cluster and single-slice CTAs,
    against the oracle's attention of every live row.  growth > 0 scales the keys of
    tile t by 1 + growth * t, so the row maxima climb tile after tile."""
    g = synth.rng(400 + N + k_max + growth)
    dq, dkv = n_q * hd, n_kv * hd
    Q = synth.round_bf16(g.standard_normal((Bq * k_max, dq), dtype=np.float32))
    kscale = (1.0 + growth * (np.arange(N) // 128)).astype(np.float32)[None, :, None]
    K = synth.round_bf16(g.standard_normal((Bq, N, dkv), dtype=np.float32) * kscale)
    V = synth.round_bf16(g.standard_normal((Bq, N, dkv), dtype=np.float32))
    idx = np.full((Bq, N), -1, np.int32)
    cnt = np.zeros(Bq, np.int32)
    for b in range(Bq):
        nb = max(1, live - 3 * b)
        idx[b, :nb] = np.sort(g.permutation(N)[:nb])
        cnt[b] = nb
    A = B.dllm_attention(to_dev(Q, torch.bfloat16), to_dev(K.reshape(Bq, N, n_kv, hd), torch.bfloat16),
                         to_dev(V.reshape(Bq, N, n_kv, hd), torch.bfloat16), to_dev(idx), to_dev(cnt), k_max)
    A = to_np(A)
    L = orc.Layer({"w_q": np.zeros((dq, dq), np.float32), "w_k": np.zeros((dkv, dq), np.float32),
                   "w_v": np.zeros((dkv, dq), np.float32), "w_o": np.zeros((dq, dq), np.float32),
                   "w_g": np.zeros((32, dq), np.float32), "w_u": np.zeros((32, dq), np.float32),
                   "w_d": np.zeros((dq, 32), np.float32), "gamma1": np.ones(dq, np.float32),
                   "gamma2": np.ones(dq, np.float32)}, n_q, n_kv, hd)
    for b in range(Bq):
        rows = np.arange(b * k_max, b * k_max + cnt[b])
        ref = orc.attention_rows(L, Q[rows], K[b], V[b])
        assert_close_layer(A[rows], ref, "bf16", f"attention b={b}")
        dead = np.arange(b * k_max + cnt[b], (b + 1) * k_max)
        assert (A[dead] == 0).all()


# --------------------------------------------------------------------------- read-back of refreshed rows
@pytest.mark.parametrize("Bq,N,k_max,row_bytes", [(3, 50, 10, 16), (2, 333, 64, 4096 * 2), (1, 7, 7, 160)])
def test_gather_rows_bit_exact(B, Bq, N, k_max, row_bytes):
    """dllm_gather_rows packs the rows idx[b, :min(count[b], k_max)] of each sequence and
    zeros the rest; entries outside [0, N) count as not live.  Pure data movement: the
    expected array is numpy indexing of the same seeded input."""
    g = synth.rng(5000 + N + k_max)
    src = g.integers(0, 256, size=(Bq, N, row_bytes), dtype=np.uint8)
    idx = np.full((Bq, N), -1, np.int32)
    cnt = np.zeros(Bq, np.int32)
    for b in range(Bq):
        n = min(N, k_max + 2 * b)                       # count[b] may exceed k_max
        idx[b, :n] = g.permutation(N)[:n]
        cnt[b] = n
    if N > 2:
        idx[0, 1] = N + 5                               # an out-of-range entry
    dst = B.dllm_gather_rows(to_dev(src), to_dev(idx), to_dev(cnt), k_max)
    got = to_np(dst).reshape(Bq * k_max, row_bytes)
    want = np.zeros_like(got)
    for b in range(Bq):
        for s in range(min(cnt[b], k_max)):
            p = idx[b, s]
            if 0 <= p < N:
                want[b * k_max + s] = src[b, p]
    np.testing.assert_array_equal(got, want)


def test_gather_rows_n_bit_exact(B):
    """dllm_gather_rows_n packs three caches of different row sizes (a step's H_out, K and
    V rows) sharing one selection in one launch, each exactly as dllm_gather_rows packs it."""
    g = synth.rng(5100)
    Bq, N, k_max = 3, 300, 40
    srcs = [g.integers(0, 256, size=(Bq, N, rb), dtype=np.uint8) for rb in (512, 256, 4096)]
    idx = np.full((Bq, N), -1, np.int32)
    cnt = np.zeros(Bq, np.int32)
    for b in range(Bq):
        n = k_max - 7 * b
        idx[b, :n] = np.sort(g.permutation(N)[:n])
        cnt[b] = n
    d_idx, d_cnt = to_dev(idx), to_dev(cnt)
    outs = B.dllm_gather_rows_n([to_dev(x) for x in srcs], d_idx, d_cnt, k_max)
    for x, o in zip(srcs, outs):
        one = B.dllm_gather_rows(to_dev(x), d_idx, d_cnt, k_max)
        assert torch.equal(o, one)
        want = np.zeros((Bq * k_max, x.shape[2]), np.uint8)
        for b in range(Bq):
            want[b * k_max:b * k_max + cnt[b]] = x[b, idx[b, :cnt[b]]]
        np.testing.assert_array_equal(to_np(o).reshape(want.shape), want)
