"""Failure paths and out-of-range writes, checked without faulting the GPU.

* Guard bytes: every array an entry point receives sits inside a larger allocation
  whose 4 KB before and after it hold a seeded byte pattern; after the calls of one
  sparse refresh step, the one-call layer step (and the vocabulary, LM head, attention,
  GEMM, KL drift and row read-back calls) at ragged shapes, every guard must be bit-unchanged -- no kernel
  wrote past the end (or before the start) of an output, a cache or a workspace.
* Bounded waits: the library's diagnostic runs the same bounded mbarrier wait the
  pipelined kernels use on a barrier nothing completes; the wait must give up after its
  limit, the status word must report the timeout, and the context must stay usable.
"""
import numpy as np
import pytest

from sparse_kv_cache_rank_gb300 import synth
from cases import forced_rows, layer_case

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GUARD_BYTES = 4096


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from sparse_kv_cache_rank_gb300 import binding
    binding.lib()
    binding.check_status(reset=True)
    return binding


class Guarded:
    """Tensors carved from allocations with GUARD_BYTES of seeded bytes on each side."""

    def __init__(self, seed):
        self.g = synth.rng(seed)
        self.items = []

    def new(self, shape, dtype, fill=None):
        el = torch.empty((), dtype=dtype).element_size()
        n = int(np.prod(shape))
        gel = GUARD_BYTES // el
        buf = torch.empty(n + 2 * gel, dtype=dtype, device="cuda")
        pat = torch.from_numpy(self.g.integers(0, 256, size=(n + 2 * gel) * el, dtype=np.uint8)).cuda()
        buf.view(torch.uint8).copy_(pat)
        t = buf[gel:gel + n].view(shape)
        if fill is not None:
            t.copy_(fill)
        head, tail = buf[:gel].clone(), buf[gel + n:].clone()
        self.items.append((buf, gel, n, head, tail))
        return t

    def check(self):
        torch.cuda.synchronize()
        for i, (buf, gel, n, head, tail) in enumerate(self.items):
            assert torch.equal(buf[:gel].view(torch.uint8), head.view(torch.uint8)), f"array {i}: guard before"
            assert torch.equal(buf[gel + n:].view(torch.uint8), tail.view(torch.uint8)), f"array {i}: guard after"


SHAPE = synth.LayerShape("guarded", B=2, N=200, d=256, n_q=4, n_kv=2, hd=64, F=320, r=64, rho=0.25,
                         dtype="bf16", prompt=100, k_recent=4)


def test_step_writes_stay_inside_their_arrays(B, orc):
    sh = SHAPE
    bf = torch.bfloat16
    c = layer_case(orc, sh, 90)
    forced = forced_rows(sh, 91)
    k = orc.budget(sh.rho, sh.N)
    k_max = min(sh.N, k + forced.shape[1])
    G = Guarded(92)
    H = G.new((sh.B, sh.N, sh.d), bf, torch.from_numpy(c.H_cur).to(bf))
    Pt = G.new((sh.r, sh.d), bf, torch.from_numpy(c.P.T.copy()).to(bf))
    pc = G.new((sh.B, sh.N, sh.r), torch.float32, torch.from_numpy(c.pc0))
    cur = G.new((sh.B, sh.N, sh.r), torch.float32)
    drift = G.new((sh.B, sh.N), torch.float32)
    pws = G.new((max(256, int(B.lib().dllm_proxy_workspace_bytes(sh.B, sh.N, sh.d, sh.r, 1))),), torch.uint8)
    B.dllm_proxy_score(H, Pt, pc, proxy_cur=cur, drift=drift, ws=pws)
    fo = G.new(forced.shape, torch.int32, torch.from_numpy(forced))
    idx = G.new((sh.B, sh.N), torch.int32)
    cnt = G.new((sh.B,), torch.int32)
    B.dllm_select_topk(drift, fo, k, idx=idx, count=cnt)
    layer = B.dllm_pack_layer({n: torch.from_numpy(v).to(bf).cuda() for n, v in c.w.items()}, sh.n_q, sh.n_kv,
                              sh.hd, eps=sh.eps, rope_theta=sh.rope_theta)
    K = G.new((sh.B, sh.N, sh.n_kv, sh.hd), bf, torch.from_numpy(c.K0.reshape(sh.B, sh.N, sh.n_kv, sh.hd)).to(bf))
    V = G.new((sh.B, sh.N, sh.n_kv, sh.hd), bf, torch.from_numpy(c.V0.reshape(sh.B, sh.N, sh.n_kv, sh.hd)).to(bf))
    O = G.new((sh.B, sh.N, sh.d), bf, torch.from_numpy(c.O0).to(bf))
    rws = G.new((B.dllm_refresh_workspace_bytes(layer, sh.B, sh.N, k_max),), torch.uint8)
    B.dllm_sparse_layer_refresh(layer, H, idx, cnt, k_max, K, V, O, pc, cur, ws=rws)
    # the one-call layer step (proxy, fused selection + gather, stream-K projections)
    lws = G.new((int(B.dllm_layer_step_workspace_bytes(layer, sh.B, sh.N, sh.r, forced.shape[1], k)),), torch.uint8)
    idx2 = G.new((sh.B, sh.N), torch.int32)
    cnt2 = G.new((sh.B,), torch.int32)
    B.dllm_layer_step(layer, Pt, H, pc, cur, drift, fo, k, idx2, cnt2, K, V, O, ws=lws)
    # attention alone over ragged live rows, and the read-back of the refreshed rows
    Q = G.new((sh.B * k_max, sh.d_q), bf, torch.randn((sh.B * k_max, sh.d_q)).to(bf))
    A = G.new((sh.B * k_max, sh.d_q), bf)
    B.dllm_attention(Q, K, V, idx, cnt, k_max, A=A)
    rows = G.new((sh.B * k_max, sh.d), bf)
    B.dllm_gather_rows(O, idx, cnt, k_max, rows)
    # plain GEMM with a ragged token count and a K split
    X = G.new((37, 192), bf, torch.randn((37, 192)).to(bf))
    W = G.new((96, 192), bf, torch.randn((96, 192)).to(bf))
    out = G.new((37, 96), torch.float32)
    B.dllm_gemm_bf16(X, W, out=out, splits=2)
    # vocabulary step, fused LM head (ragged last vocabulary tile), KL drift
    Bq, M, Vv, d = 2, 24, 4160, 256
    logits = G.new((Bq, M, Vv), torch.float32, torch.from_numpy(synth.commit_logits(Bq, M, Vv, 93)))
    valid = G.new((Bq, M), torch.uint8, torch.ones((Bq, M), dtype=torch.uint8))
    outs = (G.new((Bq, M), torch.int32), G.new((Bq, M), torch.float32), G.new((Bq, M), torch.float32),
            G.new((Bq,), torch.float32), G.new((Bq,), torch.int32))
    cws = G.new((int(B.lib().dllm_commit_workspace_bytes(Bq, M, Vv)),), torch.uint8)
    B.dllm_commit_entropy(logits, valid, out=outs, ws=cws)
    Xl = G.new((Bq * M, d), bf, torch.randn((Bq * M, d)).to(bf))
    Wl = G.new((Vv, d), bf, (torch.randn((Vv, d)) * 0.05).to(bf))
    outs2 = (G.new((Bq, M), torch.int32), G.new((Bq, M), torch.float32), G.new((Bq, M), torch.float32),
             G.new((Bq,), torch.float32), G.new((Bq,), torch.int32))
    lws = G.new((int(B.lib().dllm_lmhead_workspace_bytes(Bq, M, Vv)),), torch.uint8)
    B.dllm_lmhead_commit(Xl, Wl, valid, out=outs2, ws=lws)
    kl = G.new((sh.B, sh.N), torch.float32)
    kws = G.new((int(B.lib().dllm_kl_drift_workspace_bytes(sh.B, sh.N)),), torch.uint8)
    B.dllm_kl_drift(cur, pc, drift=kl, ws=kws)
    assert B.check_status() == 0
    G.check()


def test_bounded_wait_gives_up_and_reports(B):
    """The wait that replaces traps: it runs out on a barrier nothing completes, every
    waiting thread returns, the status word carries the timeout bit, and the next call
    on the same context works."""
    gave_up, rc, bits = B.dllm_check_wait_timeout()
    assert gave_up == 64
    assert rc == -5 and bits & B.STATUS_TIMEOUT
    x = torch.ones(1 << 20, device="cuda", dtype=torch.float32)
    assert float(x.sum().item()) == float(1 << 20)
    assert B.check_status() == 0          # cleared by the diagnostic's read
