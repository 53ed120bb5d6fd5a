"""The denoising step around the layers (EntropyCache, "How EntropyCache works",
steps 1-3) through the C ABI: token embedding, final RMSNorm of the block rows, LM
head and the commit rule; a full step of a small multi-layer stack against the
oracle's dense forward; and a sparse step of a multi-layer stack -- per-layer budgets
from the piecewise-Gaussian rho(l) (SPA-Cache, "2. Adaptive budget allocation"), the
forced block and recent rows, a drifted layer-0 input -- against the oracle run layer
by layer on its own values.

Every input comes from the seeded generators (weights, embeddings, tokens, hidden
states, caches built by the oracle); the oracle never receives a value the GPU
computed.
"""
import numpy as np
import pytest

from sparse_kv_cache_rank_gb300 import synth
from cases import (BF16_MAX_REL, FP32_REDUCTION_RTOL, assert_close_layer, assert_drift_close,
                   assert_update_close, normwise_rel, softmax_stats_bound, to_dev, to_np)

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


def test_embed_rows_and_final_norm(B, orc):
    g = synth.rng(60)
    V, d, Bq, N = 97, 128, 2, 40
    E = synth.round_bf16(g.standard_normal((V, d), dtype=np.float32))
    tok = g.integers(-2, V + 2, size=(Bq, N)).astype(np.int32)      # includes invalid ids
    H = torch.full((Bq, N, d), 7.0, dtype=torch.bfloat16, device="cuda")
    B.dllm_embed(to_dev(E, torch.bfloat16), to_dev(tok), H)
    want = np.where(((tok >= 0) & (tok < V))[..., None], E[np.clip(tok, 0, V - 1)], 0.0).astype(np.float32)
    np.testing.assert_array_equal(to_np(H), want)
    rows = np.array([[3, 39, -1, 0], [5, 5, 40, 17]], np.int32)       # -1 / N give zero rows
    H2 = torch.zeros((Bq, N, d), dtype=torch.bfloat16, device="cuda")
    B.dllm_embed(to_dev(E, torch.bfloat16), to_dev(tok), H2, rows=to_dev(rows))
    got = to_np(H2)
    for b in range(Bq):
        for p in range(N):
            exp = want[b, p] if p in rows[b] else 0.0
            np.testing.assert_array_equal(got[b, p], exp)
    gamma = synth.round_bf16((0.5 + g.random(d)).astype(np.float32))
    out = to_np(B.dllm_rows_rmsnorm(H, to_dev(rows), to_dev(gamma, torch.bfloat16), 1e-5))
    for b in range(Bq):
        for j, p in enumerate(rows[b]):
            o = out[b * 4 + j]
            if 0 <= p < N:     # the oracle normalises the seeded row itself
                ref = orc.lmhead(want[b, p][None], gamma, np.eye(d, dtype=np.float32))[0]
                assert_close_layer(o, ref, "bf16", "final norm")
            else:
                assert (o == 0).all()


def _stats_against_oracle(orc, conf, ent, logits_g, logits_ref, live):
    """GPU confidence / entropy against the oracle's statistics of its own logits, within
    what the GPU logits' measured error can move them (cases.softmax_stats_bound)."""
    assert_close_layer(logits_g, logits_ref, "bf16", "logits")
    delta = float(np.abs(np.asarray(logits_g, np.float64) - logits_ref).max())
    _, pm, H = orc.vocab_stats(logits_ref)
    dc, dh = softmax_stats_bound(logits_ref, delta)
    assert (np.abs(conf - pm)[live] <= dc[live] + FP32_REDUCTION_RTOL * pm[live]).all()
    assert (np.abs(ent - H)[live] <= dh[live] + FP32_REDUCTION_RTOL * H[live] + 1e-6).all()
    return pm, H


def test_lmhead_and_commit_parity(B, orc):
    g = synth.rng(61)
    d, V, M = 512, 4096, 32
    h = synth.round_bf16(g.standard_normal((1, M, d), dtype=np.float32))
    W = synth.round_bf16((g.standard_normal((V, d)) * 0.1).astype(np.float32))
    gamma = np.ones(d, np.float32)
    rows = np.arange(M, dtype=np.int32)[None]
    X = B.dllm_rows_rmsnorm(to_dev(h, torch.bfloat16), to_dev(rows), to_dev(gamma, torch.bfloat16))
    logits = B.dllm_gemm_bf16(X, to_dev(W, torch.bfloat16)).view(1, M, V)
    ref = orc.lmhead(h[0], gamma, W)
    valid = np.ones((1, M), np.uint8)
    tok, conf, ent, E, full = B.dllm_commit_entropy(logits, to_dev(valid))
    live = valid.astype(bool)[0]
    pm, H = _stats_against_oracle(orc, to_np(conf)[0], to_np(ent)[0], to_np(logits)[0], ref, live)
    # the decision: these logits put every confidence far below 0.9, so the rule commits
    # the single most confident row; where the oracle's top row stays on top under the
    # logits' error, the GPU commits that row alone, with the oracle's token when the
    # row's top two logits are further apart than the error can close
    delta = float(np.abs(to_np(logits)[0] - ref).max())
    dc, _ = softmax_stats_bound(ref, delta)
    assert (pm + dc < 0.9).all()
    order = np.argsort(-pm)
    t = to_np(tok)[0]
    if pm[order[0]] - dc[order[0]] > pm[order[1]] + dc[order[1]]:
        row = order[0]
        assert (np.delete(t, row) == -1).all() and t[row] >= 0
        top2 = np.sort(ref[row])[-2:]
        if top2[1] - top2[0] > 2 * delta:
            assert t[row] == ref[row].argmax()


@pytest.mark.parametrize("Bq,M,V,d,scale", [(1, 32, 4096, 512, 0.1), (2, 24, 4160, 256, 0.5),
                                             (1, 32, 126464, 512, 0.05), (2, 8, 1024, 128, 3.0)])
def test_lmhead_commit_fused(B, orc, Bq, M, V, d, scale):
    """The LM head fused with the vocabulary statistics gives the unfused path's results
    (tokens exactly, confidence and entropy within the fp32 reduction tolerance), with
    invalid rows, a ragged last vocabulary tile (V = 4160) and the LLaDA vocabulary; and
    both agree with the oracle's statistics of its own logits within what the logits'
    bf16 error can move them."""
    g = synth.rng(71 + M + V)
    X = synth.round_bf16(g.standard_normal((Bq * M, d), dtype=np.float32))
    W = synth.round_bf16((g.standard_normal((V, d)) * scale / np.sqrt(d) * 8).astype(np.float32))
    valid = (g.random((Bq, M)) > 0.2).astype(np.uint8)
    valid[:, 0] = 1
    Xd, Wd, vd = to_dev(X, torch.bfloat16), to_dev(W, torch.bfloat16), to_dev(valid)
    logits = B.dllm_gemm_bf16(Xd, Wd).view(Bq, M, V)
    tok_u, conf_u, ent_u, E_u, full_u = B.dllm_commit_entropy(logits, vd)
    tok, conf, ent, E, full = B.dllm_lmhead_commit(Xd, Wd, vd)
    live = valid.astype(bool)
    np.testing.assert_allclose(to_np(conf)[live], to_np(conf_u)[live], rtol=FP32_REDUCTION_RTOL, atol=1e-9)
    np.testing.assert_allclose(to_np(ent)[live], to_np(ent_u)[live], rtol=FP32_REDUCTION_RTOL, atol=1e-6)
    np.testing.assert_array_equal(to_np(tok), to_np(tok_u))
    ref = np.stack([X[b * M:(b + 1) * M].astype(np.float64) @ W.T.astype(np.float64) for b in range(Bq)])
    _stats_against_oracle(orc, to_np(conf), to_np(ent), to_np(logits), ref, live)
    again = B.dllm_lmhead_commit(Xd, Wd, vd)
    assert all(torch.equal(a, b) for a, b in zip(again, (tok, conf, ent, E, full)))


# --------------------------------------------------------------------------- stacks
TINY_STACK = synth.LayerShape("tiny-stack", B=1, N=96, d=256, n_q=4, n_kv=2, hd=64, F=256, r=64,
                              rho=0.25, dtype="bf16", V=512, prompt=64, block=32, layers=2)


def _seeded_stack(B, orc, sh, seed, rho=None, k_recent=4, **kw):
    """A DecodeStack whose weights, proxies, embedding, LM head and prompt come from the
    seeded generators; returns (stack, numpy inputs for the oracle)."""
    from sparse_kv_cache_rank_gb300.stack import DecodeStack
    bf = torch.bfloat16
    ws = [synth.layer_weights(sh, seed + l) for l in range(sh.layers)]
    Ps = [synth.round_bf16(orc.proxy_matrix(w["w_v"], w["gamma1"], sh.r).astype(np.float32)) for w in ws]
    g = synth.rng(seed + 100)
    E = synth.round_bf16((g.standard_normal((sh.V, sh.d)) * 0.02).astype(np.float32))
    W_lm = synth.round_bf16((g.standard_normal((sh.V, sh.d)) * 0.02).astype(np.float32))
    prompt = g.integers(0, sh.V - 1, size=(sh.B, sh.prompt)).astype(np.int32)
    st = DecodeStack(sh, seed, torch.device("cuda"), rho=rho, k_recent=k_recent,
                     weights=[{n: to_dev(v, bf) for n, v in w.items()} for w in ws],
                     proxies=[to_dev(P.T.copy(), bf) for P in Ps], embedding=to_dev(E, bf),
                     lm_head=to_dev(W_lm, bf), prompt_tokens=to_dev(prompt), **kw)
    tokens = np.full((sh.B, sh.N), sh.V - 1, np.int32)
    tokens[:, :sh.prompt] = prompt
    Ls = [orc.Layer(w, sh.n_q, sh.n_kv, sh.hd, eps=sh.eps, rope_theta=sh.rope_theta) for w in ws]
    return st, dict(w=ws, P=Ps, L=Ls, E=E, W_lm=W_lm, tokens=tokens)


def test_full_step_equals_dense_forward(B, orc):
    """A full step of the stack equals the oracle's dense forward through every layer
    followed by the final norm and the LM head of the block rows."""
    sh = TINY_STACK
    st, o = _seeded_stack(B, orc, sh, 62, keep_logits=True)
    st.forward(True)
    torch.cuda.synchronize()
    H = o["E"][o["tokens"]]                   # the embedding of the seeded tokens
    for L in o["L"]:
        _, _, H = orc.layer_full(L, H)
        H = synth.round_bf16(H)               # the cache stores bf16 hidden states between layers
    rows = np.arange(sh.prompt, sh.prompt + sh.block)
    ref = orc.lmhead(H[0, rows], np.ones(sh.d, np.float32), o["W_lm"])
    assert_close_layer(to_np(st.logits)[0], ref, "bf16", "logits after 2 layers")
    assert_close_layer(to_np(st.layers[-1].O), H, "bf16", "last layer output")


CHAIN = synth.LayerShape("chain", B=2, N=160, d=256, n_q=4, n_kv=2, hd=64, F=320, r=64, rho=0.0,
                         dtype="bf16", V=512, prompt=96, block=32, layers=3, k_recent=4)
CHAIN_RHO = dict(base=0.02, peak=0.06, centre=0.0, sigma_left=1.2, sigma_right=1.2)


def test_sparse_stack_step_chained(B, orc):
    """One partial denoising step of a 3-layer stack: every layer scores its input against
    its cached proxies, selects its rho(l) budget (10, 8, 5 rows of 160) on top of the
    forced rows (the block's masked positions and the 4 recent ones) and refreshes them;
    each layer's input is the previous layer's refreshed output cache.  The oracle runs
    the same step layer by layer on its own values from the same seeded state, and at
    every layer the drift, the selection, K/V/H_out of the refreshed rows, the untouched
    rows and the cached proxies are compared.

    The layer-0 input moves 12 rows per sequence by graded amounts (a geometric ladder,
    synth.hidden_ladder) and leaves the rest unchanged, so that each budget boundary falls
    between rungs whose drifts differ by far more than the bf16 rounding a layer passes
    on to the next (checked below on the oracle's drifts); rows whose input did not change
    have zero drift and are never drift-selected (the eligibility threshold)."""
    from sparse_kv_cache_rank_gb300.stack import RhoSchedule
    sh = CHAIN
    st, o = _seeded_stack(B, orc, sh, 500, rho=RhoSchedule(**CHAIN_RHO), k_recent=sh.k_recent)
    g = synth.rng(510)
    H_prev = synth.round_bf16(g.standard_normal((sh.B, sh.N, sh.d), dtype=np.float32))
    # step t-1: every layer's caches from the oracle's dense forward, given to both sides
    caches, X = [], H_prev
    for l, L in enumerate(o["L"]):
        K, V, O = (synth.round_bf16(a) for a in orc.layer_full(L, X))
        pc, _ = orc.proxy_score(X, o["P"][l], np.ones((sh.B, sh.N, sh.r), np.float32))
        caches.append((K, V, O, pc))
        lay = st.layers[l]
        lay.K.copy_(to_dev(K.reshape(sh.B, sh.N, sh.n_kv, sh.hd), torch.bfloat16))
        lay.V.copy_(to_dev(V.reshape(sh.B, sh.N, sh.n_kv, sh.hd), torch.bfloat16))
        lay.O.copy_(to_dev(O, torch.bfloat16))
        lay.pc.copy_(to_dev(pc))
        X = O
    masked, recent = synth.block_layout(sh, 501)
    forced = np.full((sh.B, sh.block + sh.k_recent), -1, np.int32)
    forced[:, :masked.shape[1] + recent.shape[1]] = np.concatenate([masked, recent], 1)
    st.forced.copy_(to_dev(forced))
    H_cur = synth.hidden_ladder(sh, H_prev, forced, 511)

    rec = []
    st.forward(False, H0=to_dev(H_cur, torch.bfloat16), record=rec)
    torch.cuda.synchronize()
    assert B.check_status() == 0

    X, X_g = H_cur, H_cur
    for l, L in enumerate(o["L"]):
        k = orc.budget(orc.rho(l, **CHAIN_RHO), sh.N)
        assert k == st.budgets[l] and k == (10, 8, 5)[l]
        K0, V0, O0, pc0 = caches[l]
        cur_o, drift_o = orc.proxy_score(X, o["P"][l], pc0)
        idx_o, cnt_o = orc.select_topk(drift_o, forced, k)
        for b in range(sh.B):     # no near-tie at the boundary: the next rung is >= 20 % lower
            fs = set(forced[b].tolist())
            el = np.sort([drift_o[b, i] for i in range(sh.N) if i not in fs and drift_o[b, i] > 1e-6])[::-1]
            assert len(el) > k and el[k - 1] - el[k] >= 0.2 * el[k - 1], (l, b, el[:k + 1])
        d_g = to_np(rec[l]["drift"])
        if l == 0:
            assert_drift_close(d_g, drift_o)
        unchanged = drift_o == 0           # input identical to the one the cache holds
        assert (d_g[unchanged] <= 1e-6).all()
        np.testing.assert_array_equal(to_np(rec[l]["cnt"]), cnt_o)
        np.testing.assert_array_equal(to_np(rec[l]["idx"]), idx_o)
        Ko, Vo, Oo, pco = K0.copy(), V0.copy(), O0.copy(), pc0.copy()
        orc.layer_refresh(L, X, idx_o, cnt_o, Ko, Vo, Oo, pco, cur_o)
        lay = st.layers[l]
        Kg = to_np(lay.K).reshape(sh.B, sh.N, sh.d_kv)
        Vg = to_np(lay.V).reshape(sh.B, sh.N, sh.d_kv)
        Og, pcg = to_np(lay.O), to_np(lay.pc)
        for b in range(sh.B):
            I = idx_o[b, :cnt_o[b]]
            rest = np.setdiff1d(np.arange(sh.N), I)
            for name, got, ref in (("K", Kg, K0), ("V", Vg, V0), ("O", Og, O0), ("pc", pcg, pc0)):
                np.testing.assert_array_equal(got[b, rest], ref[b, rest], err_msg=f"layer {l} {name}")
            assert_close_layer(Kg[b, I], Ko[b, I], "bf16", f"layer {l} K b={b}")
            assert_close_layer(Vg[b, I], Vo[b, I], "bf16", f"layer {l} V b={b}")
            assert_close_layer(Og[b, I], Oo[b, I], "bf16", f"layer {l} H_out b={b}")
            assert_update_close(Og[b, I], Oo[b, I], X_g[b, I], "bf16", f"layer {l} update b={b}",
                                h_in_ref=X[b, I])
            # proxies of this step: same inputs at layer 0, bf16-close inputs deeper down
            tol = FP32_REDUCTION_RTOL if l == 0 else BF16_MAX_REL
            assert normwise_rel(pcg[b, I], pco[b, I]) < tol
        X, X_g = synth.round_bf16(Oo), Og


def test_graph_step_equals_eager(B, orc):
    """A partial step replayed from a captured CUDA graph gives the eager step's outputs
    bit for bit (same kernels, fixed reduction orders) from the same state."""
    from sparse_kv_cache_rank_gb300.stack import RhoSchedule
    sh = CHAIN
    st, _ = _seeded_stack(B, orc, sh, 520, rho=RhoSchedule(**CHAIN_RHO), k_recent=sh.k_recent)
    st.prefill()
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    st.H0.add_((torch.randn(st.H0.shape, generator=g, device="cuda") * 0.3).to(st.H0.dtype))
    state = [t.clone() for L in st.layers for t in (L.K, L.V, L.O)] + [st.pc_all.clone()]

    def restore():
        ts = [t for L in st.layers for t in (L.K, L.V, L.O)] + [st.pc_all]
        for t, s in zip(ts, state):
            t.copy_(s)

    outs = st.forward(False)
    eager = [t.clone() for t in outs] + [t.clone() for L in st.layers for t in (L.K, L.V, L.O)]
    restore()
    gr = st.graph(lambda: st.forward(False), warmup=1)
    restore()
    gr.replay()
    torch.cuda.synchronize()
    graphed = [t.clone() for t in st.out] + [t.clone() for L in st.layers for t in (L.K, L.V, L.O)]
    assert all(torch.equal(a, b) for a, b in zip(eager, graphed))
    assert B.check_status() == 0


def test_decode_loop_commits_and_advances(B):
    """Rule-driven decoding of the tiny stack, with the steps replayed from captured CUDA
    graphs: at least one token per step, history of the k most recent decoded positions,
    blocks advance, every position decoded at the end."""
    from sparse_kv_cache_rank_gb300.stack import DecodeStack
    sh = TINY_STACK
    st = DecodeStack(sh, 63, torch.device("cuda"), k_recent=4)
    st.capture()
    st.prefill()
    steps = 0
    while not st.done() and steps < 200:
        assert st.decode_step() >= 1
        steps += 1
        assert all(len(h) <= 4 for h in st.history)
    assert st.done()
    assert steps <= sh.N - sh.prompt
    B.check_status()


def test_forced_sparse_steps_run(B):
    """Sparse steps (the rule overridden) refresh the forced rows plus at most k_l rows per layer."""
    from sparse_kv_cache_rank_gb300.stack import DecodeStack
    sh = TINY_STACK
    st = DecodeStack(sh, 64, torch.device("cuda"), k_recent=4)
    st.prefill()
    counts = st.rows_per_layer(False)
    F = int((st.forced >= 0).sum().item())
    for l, c in enumerate(counts):
        assert F <= c <= F + st.budgets[l]
    for _ in range(3):
        st.decode_step(force_sparse=True)
    B.check_status()
