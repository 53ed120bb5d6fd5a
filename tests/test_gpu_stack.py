"""The denoising step around the layers (EntropyCache, "How EntropyCache works",
steps 1-3) through the C ABI: token embedding, final RMSNorm of the block rows, LM
head and the commit rule; and a full step of a small multi-layer stack against the
oracle's dense forward of every layer followed by its LM head."""
import numpy as np
import pytest

from sparse_kv_cache_rank_gb300 import synth
from cases import FP32_REDUCTION_RTOL, assert_close_layer, normwise_rel, to_dev, to_np

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_kv_cache_rank_gb300 import binding
    binding.lib()
    return binding


def test_embed_rows_and_final_norm(B, orc):
    g = synth.rng(60)
    V, d, Bq, N = 97, 128, 2, 40
    E = synth.round_bf16(g.standard_normal((V, d), dtype=np.float32))
    tok = g.integers(-2, V + 2, size=(Bq, N)).astype(np.int32)      # includes invalid ids
    H = torch.full((Bq, N, d), 7.0, dtype=torch.bfloat16, device="cuda")
    B.dllm_embed(to_dev(E, torch.bfloat16), to_dev(tok), H)
    want = np.where(((tok >= 0) & (tok < V))[..., None], E[np.clip(tok, 0, V - 1)], 0.0)
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
    out = B.dllm_rows_rmsnorm(H, to_dev(rows), to_dev(gamma, torch.bfloat16), 1e-5)
    h = to_np(H)
    for b in range(Bq):
        for j, p in enumerate(rows[b]):
            o = to_np(out)[b * 4 + j]
            if 0 <= p < N:
                ref = orc.lmhead(h[b, p][None], gamma, np.eye(d, dtype=np.float32))[0]
                assert_close_layer(o, ref, "bf16", "final norm")
            else:
                assert (o == 0).all()


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
    assert_close_layer(to_np(logits)[0], ref, "bf16", "logits")
    valid = np.ones((1, M), np.uint8)
    tok, conf, ent, E, full = B.dllm_commit_entropy(logits, to_dev(valid))
    am, pm, H = orc.vocab_stats(to_np(logits))      # oracle statistics of the GPU's logits
    np.testing.assert_allclose(to_np(conf), pm, rtol=FP32_REDUCTION_RTOL, atol=1e-9)
    np.testing.assert_allclose(to_np(ent), H, rtol=FP32_REDUCTION_RTOL, atol=1e-6)
    t_o, E_o, f_o = orc.commit_rule(am, to_np(conf), to_np(ent), valid)
    np.testing.assert_array_equal(to_np(tok), t_o)
    np.testing.assert_array_equal(to_np(full), f_o)


@pytest.mark.parametrize("Bq,M,V,d,scale", [(1, 32, 4096, 512, 0.1), (2, 24, 4160, 256, 0.5),
                                             (1, 32, 126464, 512, 0.05), (2, 8, 1024, 128, 3.0)])
def test_lmhead_commit_fused(B, orc, Bq, M, V, d, scale):
    """The LM head fused with the vocabulary statistics gives the unfused path's decisions:
    argmax and committed tokens exactly, confidence and entropy within the fp32 reduction
    tolerance (against the oracle's statistics of the same logits), with invalid rows, a
    ragged last vocabulary tile (V = 4160) and the LLaDA vocabulary."""
    g = synth.rng(71 + M + V)
    X = synth.round_bf16(g.standard_normal((Bq * M, d), dtype=np.float32))
    W = synth.round_bf16((g.standard_normal((V, d)) * scale / np.sqrt(d) * 8).astype(np.float32))
    valid = (g.random((Bq, M)) > 0.2).astype(np.uint8)
    valid[:, 0] = 1
    Xd, Wd, vd = to_dev(X, torch.bfloat16), to_dev(W, torch.bfloat16), to_dev(valid)
    logits = B.dllm_gemm_bf16(Xd, Wd).view(Bq, M, V)
    tok_u, conf_u, ent_u, E_u, full_u = B.dllm_commit_entropy(logits, vd)
    tok, conf, ent, E, full = B.dllm_lmhead_commit(Xd, Wd, vd)
    am, pm, H = orc.vocab_stats(to_np(logits))
    live = valid.astype(bool)
    np.testing.assert_allclose(to_np(conf)[live], pm[live], rtol=FP32_REDUCTION_RTOL, atol=1e-9)
    np.testing.assert_allclose(to_np(ent)[live], H[live], rtol=FP32_REDUCTION_RTOL, atol=1e-6)
    t_o, E_o, f_o = orc.commit_rule(am, to_np(conf), to_np(ent), valid)
    np.testing.assert_array_equal(to_np(tok), t_o)
    np.testing.assert_array_equal(to_np(full), f_o)
    np.testing.assert_array_equal(to_np(tok), to_np(tok_u))
    again = B.dllm_lmhead_commit(Xd, Wd, vd)
    assert all(torch.equal(a, b) for a, b in zip(again, (tok, conf, ent, E, full)))


TINY_STACK = synth.LayerShape("tiny-stack", B=1, N=96, d=256, n_q=4, n_kv=2, hd=64, F=256, r=64,
                              rho=0.25, dtype="bf16", V=512, prompt=64, block=32, layers=2)


def test_full_step_equals_dense_forward(B, orc):
    """A full step of the stack equals the oracle's dense forward through every layer
    followed by the final norm and the LM head of the block rows."""
    from sparse_kv_cache_rank_gb300.stack import DecodeStack
    sh = TINY_STACK
    st = DecodeStack(sh, 62, torch.device("cuda"), k_recent=4, keep_weights=True, proxy_method="svd",
                     keep_logits=True)
    st.forward(True)
    torch.cuda.synchronize()
    H = to_np(st.H0)
    for w in st.weights:
        L = orc.Layer({k: to_np(v) for k, v in w.items()}, sh.n_q, sh.n_kv, sh.hd)
        _, _, H = orc.layer_full(L, H)
        H = synth.round_bf16(H)           # the cache stores bf16 hidden states between layers
    rows = np.arange(sh.prompt, sh.prompt + sh.block)
    ref = orc.lmhead(H[0, rows], to_np(st.gamma_f), to_np(st.W_lm))
    assert_close_layer(to_np(st.logits)[0], ref, "bf16", "logits after 2 layers")
    assert_close_layer(to_np(st.layers[-1].O), H, "bf16", "last layer output")


def test_decode_loop_commits_and_advances(B):
    """Rule-driven decoding of the tiny stack: at least one token per step, history of the
    k most recent decoded positions, blocks advance, every position decoded at the end."""
    from sparse_kv_cache_rank_gb300.stack import DecodeStack
    sh = TINY_STACK
    st = DecodeStack(sh, 63, torch.device("cuda"), k_recent=4)
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
    counts = st.count_rows(False)
    F = int((st.forced >= 0).sum().item())
    for l, c in enumerate(counts):
        assert F <= c <= F + st.budgets[l]
    for _ in range(3):
        st.decode_step(force_sparse=True)
    B.check_status()
