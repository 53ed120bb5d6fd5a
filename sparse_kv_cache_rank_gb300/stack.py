"""A multi-layer denoising model driven through the C ABI.

One denoising step (EntropyCache, "How EntropyCache works"):
  1. forward: every layer either recomputes all rows (full step) or runs the sparse
     refresh of SPA-Cache ("1. Update identification via singular proxy",
     "2. Adaptive budget allocation", "3. Sparse execution"): proxy drift of the
     layer input, top-k_l rows with k_l = ceil(rho(l) N), plus the always-recomputed
     rows (masked tokens of the current block and the k most recently decoded ones);
  2. decode: final RMSNorm of the block rows, LM head, softmax statistics, threshold
     commit, maximum entropy E of the newly decoded tokens;
  3. decide: E > tau -> the next step is a full forward, else partial.
The host keeps the token ids, the block pointer and the decode history; the device
does every step of the computation (library kernels).  Unless given, weights are
random N(0, 0.02) from a seeded generator (no trained checkpoint exists here).

Every buffer a step touches is allocated once, here, so a whole step (all layers, the
LM head and the commit) can be captured in one CUDA graph and replayed: the host then
issues one graph launch per step instead of three binding calls and about ten kernel
launches per layer (`capture`).
"""
from __future__ import annotations

import dataclasses
from collections import deque

import torch

from . import binding as B
from .proxy_setup import build_proxy_matrix
from .synth import LayerShape


@dataclasses.dataclass
class RhoSchedule:
    """Piecewise Gaussian update ratio over depth (SPA-Cache, "2. Adaptive budget allocation")."""
    base: float = 0.05
    peak: float = 0.30
    centre: float = 16.0
    sigma_left: float = 6.0
    sigma_right: float = 6.0

    def rho(self, l: int) -> float:
        return B.dllm_layer_rho(l, self.base, self.peak, self.centre, self.sigma_left, self.sigma_right)


class _Layer:
    def __init__(self, layer, Pt, K, V, O, pc, cur):
        self.layer, self.Pt, self.K, self.V, self.O, self.pc, self.cur = layer, Pt, K, V, O, pc, cur


class DecodeStack:
    """weights: optional list (one per layer) of dicts of device tensors in nn.Linear layout
    (w_q, w_k, w_v, w_o, w_g, w_u, w_d, gamma1, gamma2); proxies: optional list of the
    layers' Pt [r, d]; embedding / lm_head: optional [V, d] tensors; prompt_tokens:
    optional [B, prompt] int32.  What is not given is drawn from `seed`."""

    def __init__(self, shape: LayerShape, seed: int, device, rho: RhoSchedule | None = None,
                 uniform_rho: float | None = None, k_recent: int = 8, conf_thresh: float = 0.9,
                 tau: float = 2.0, proxy_method: str = "gram", keep_weights: bool = False,
                 keep_logits: bool = False, weights=None, proxies=None, embedding=None, lm_head=None,
                 prompt_tokens=None):
        self.sh = sh = shape
        self.dev = device
        self.rho = rho or RhoSchedule()
        self.uniform_rho = uniform_rho
        self.k_recent = k_recent
        self.conf_thresh, self.tau = conf_thresh, tau
        bf = torch.bfloat16
        gen = torch.Generator(device=device)
        gen.manual_seed(seed)

        def randn(*s, std=1.0):
            return (torch.randn(s, generator=gen, device=device, dtype=torch.float32) * std).to(bf)

        d, dq, dkv, F, Bn, N = sh.d, sh.d_q, sh.d_kv, sh.F, sh.B, sh.N
        nl = sh.layers
        self.layers = []
        self.weights = [] if keep_weights else None
        self.keep_logits = keep_logits   # materialise the block's logits (else the fused LM head)
        self.logits = None
        # proxies of every layer in one allocation each, so a caller can save or restore
        # all layers' proxy caches with one copy
        self.pc_all = torch.zeros((nl, Bn, N, sh.r), device=device, dtype=torch.float32)
        self.cur_all = torch.zeros_like(self.pc_all)
        for l in range(nl):
            if weights is not None:
                w = weights[l]
            else:
                w = {"w_q": randn(dq, d, std=0.02), "w_k": randn(dkv, d, std=0.02),
                     "w_v": randn(dkv, d, std=0.02), "w_o": randn(d, dq, std=0.02),
                     "w_g": randn(F, d, std=0.02), "w_u": randn(F, d, std=0.02), "w_d": randn(d, F, std=0.02),
                     "gamma1": torch.ones(d, device=device, dtype=bf),
                     "gamma2": torch.ones(d, device=device, dtype=bf)}
            layer = B.dllm_pack_layer(w, sh.n_q, sh.n_kv, sh.hd, eps=sh.eps, rope_theta=sh.rope_theta)
            if proxies is not None:
                Pt = proxies[l].contiguous()
            else:
                Pt = build_proxy_matrix(w["w_v"], w["gamma1"], sh.r, method=proxy_method)
            if keep_weights:
                self.weights.append(w)
            del w
            K = torch.empty((Bn, N, sh.n_kv, sh.hd), device=device, dtype=bf)
            self.layers.append(_Layer(layer, Pt, K, torch.empty_like(K),
                                      torch.empty((Bn, N, d), device=device, dtype=bf),
                                      self.pc_all[l], self.cur_all[l]))
        self.E = embedding if embedding is not None else randn(sh.V, d, std=0.02)
        self.W_lm = lm_head if lm_head is not None else randn(sh.V, d, std=0.02)
        self.gamma_f = torch.ones(d, device=device, dtype=bf)
        self.mask_id = sh.V - 1
        # tokens: prompt ids uniform in [0, V-2], generation region masked
        self.tokens = torch.full((Bn, N), self.mask_id, dtype=torch.int32, device=device)
        if prompt_tokens is not None:
            self.tokens[:, :sh.prompt] = prompt_tokens.to(device=device, dtype=torch.int32)
        else:
            self.tokens[:, :sh.prompt] = torch.randint(0, sh.V - 1, (Bn, sh.prompt), generator=gen,
                                                       device=device, dtype=torch.int32)
        self.H0 = torch.empty((Bn, N, d), device=device, dtype=bf)
        B.dllm_embed(self.E, self.tokens, self.H0)
        self.tokens_host = self.tokens.cpu()
        self.block = 0
        self.history = [deque(maxlen=k_recent) for _ in range(Bn)]
        self.full_next = True
        # scratch and step outputs (fixed addresses, see `capture`)
        self.drift = torch.empty((Bn, N), device=device, dtype=torch.float32)
        self.idx = torch.empty((Bn, N), device=device, dtype=torch.int32)
        self.cnt = torch.empty((Bn,), device=device, dtype=torch.int32)
        self.idx_all = torch.arange(N, device=device, dtype=torch.int32).repeat(Bn, 1).contiguous()
        self.cnt_all = torch.full((Bn,), N, device=device, dtype=torch.int32)
        self.ws = torch.empty(max(B.dllm_refresh_workspace_bytes(self.layers[0].layer, Bn, N, N),
                                  B.dllm_layer_step_workspace_bytes(self.layers[0].layer, Bn, N, sh.r,
                                                                    sh.block + k_recent, N)),
                              device=device, dtype=torch.uint8)
        self.ws_proxy = torch.empty(max(256, int(B.lib().dllm_proxy_workspace_bytes(Bn, N, d, sh.r, B.DLLM_BF16))),
                                    device=device, dtype=torch.uint8)
        self.ws_lm = torch.empty(int(B.lib().dllm_lmhead_workspace_bytes(Bn, sh.block, sh.V)),
                                 device=device, dtype=torch.uint8)
        self.Xf = torch.empty((Bn * sh.block, d), device=device, dtype=bf)
        self.out = (torch.empty((Bn, sh.block), dtype=torch.int32, device=device),
                    torch.empty((Bn, sh.block), dtype=torch.float32, device=device),
                    torch.empty((Bn, sh.block), dtype=torch.float32, device=device),
                    torch.empty((Bn,), dtype=torch.float32, device=device),
                    torch.empty((Bn,), dtype=torch.int32, device=device))
        self.forced = torch.full((Bn, sh.block + k_recent), -1, dtype=torch.int32, device=device)
        self.valid = torch.zeros((Bn, sh.block), dtype=torch.uint8, device=device)
        self.block_rows = torch.zeros((Bn, sh.block), dtype=torch.int32, device=device)
        self.budgets = [self.budget(l) for l in range(nl)]
        self.graphs = {}
        self._set_block_rows()

    # ------------------------------------------------------------------ host bookkeeping
    @property
    def n_blocks(self):
        return (self.sh.N - self.sh.prompt) // self.sh.block

    def budget(self, l: int) -> int:
        r = self.uniform_rho if self.uniform_rho is not None else self.rho.rho(l)
        return B.dllm_layer_budget(r, self.sh.N)

    def _set_block_rows(self):
        sh = self.sh
        start = sh.prompt + self.block * sh.block
        pos = torch.arange(start, start + sh.block, dtype=torch.int32)
        self.block_rows.copy_(pos.repeat(sh.B, 1))
        self._refresh_forced()

    def _refresh_forced(self):
        """Masked positions of the current block plus the k most recently decoded ones
        (written into the fixed device buffers `forced` and `valid`)."""
        sh = self.sh
        start = sh.prompt + self.block * sh.block
        rows = []
        valid = []
        for b in range(sh.B):
            blk = self.tokens_host[b, start:start + sh.block]
            masked = (blk == self.mask_id)
            valid.append(masked.to(torch.uint8))
            f = [start + i for i in range(sh.block) if masked[i]] + list(self.history[b])
            f += [-1] * (sh.block + self.k_recent - len(f))
            rows.append(f)
        self.forced.copy_(torch.tensor(rows, dtype=torch.int32))
        self.valid.copy_(torch.stack(valid))

    # ------------------------------------------------------------------ device step
    def forward(self, full: bool, H0=None, record: list | None = None):
        """Layers + LM head + commit on the current stream.  Returns the device tensors
        (token, conf, entropy, E, full_next).  With `record` (a list), one dict per layer
        is appended: the layer's drift, selection and row count (copies)."""
        sh = self.sh
        H = self.H0 if H0 is None else H0
        for l, L in enumerate(self.layers):
            if full:
                B.dllm_proxy_score(H, L.Pt, L.pc, proxy_cur=L.cur, drift=self.drift, ws=self.ws_proxy)
                idx, cnt = self.idx_all, self.cnt_all
                B.dllm_sparse_layer_refresh(L.layer, H, idx, cnt, sh.N, L.K, L.V, L.O, L.pc, L.cur, ws=self.ws)
            else:
                # proxy + drift, the budget's selection with the forced rows, the refresh:
                # one library call per layer
                idx, cnt = B.dllm_layer_step(L.layer, L.Pt, H, L.pc, L.cur, self.drift, self.forced,
                                             self.budgets[l], self.idx, self.cnt, L.K, L.V, L.O, ws=self.ws)
            if record is not None:
                record.append({"drift": self.drift.clone(), "idx": idx.clone(), "cnt": cnt.clone(),
                               "k": sh.N if full else self.budgets[l]})
            H = L.O
        X = B.dllm_rows_rmsnorm(H, self.block_rows, self.gamma_f, sh.eps, out=self.Xf)
        if self.keep_logits:
            logits = B.dllm_gemm_bf16(X, self.W_lm).view(sh.B, sh.block, sh.V)
            self.logits = logits
            return B.dllm_commit_entropy(logits, self.valid, self.conf_thresh, self.tau, out=self.out)
        # LM head fused with the softmax statistics (the logits are never stored)
        return B.dllm_lmhead_commit(X, self.W_lm, self.valid, self.conf_thresh, self.tau, out=self.out,
                                    ws=self.ws_lm)

    def graph(self, fn, warmup: int = 1):
        """Captures fn() (calls on this stack's fixed buffers) in a CUDA graph after
        `warmup` eager calls; returns the graph (replay() runs it on the current stream)."""
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize(self.dev)
        side = torch.cuda.Stream(self.dev)
        side.wait_stream(torch.cuda.current_stream(self.dev))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            fn()
        torch.cuda.current_stream(self.dev).wait_stream(side)
        return g

    def capture(self):
        """CUDA graphs of the full and of the partial step; `run` replays them.  A graph
        reads the token embedding H0, the forced rows, the block rows and the valid mask
        from their fixed buffers, which the host rewrites between steps."""
        if self.keep_logits:
            raise RuntimeError("capture() uses the fused LM head (keep_logits=False)")
        self.graphs = {True: self.graph(lambda: self.forward(True)),
                       False: self.graph(lambda: self.forward(False))}

    def run(self, full: bool):
        """One step: the captured graph when there is one, else the eager calls."""
        g = self.graphs.get(full)
        if g is None:
            return self.forward(full)
        g.replay()
        return self.out

    def rows_per_layer(self, full: bool):
        """Rows refreshed at each layer by one eager step (synchronises; for reporting)."""
        rec = []
        self.forward(full, record=rec)
        return [int(r["cnt"].sum().item()) for r in rec]

    # ------------------------------------------------------------------ decode loop
    def decode_step(self, force_sparse: bool = False):
        """One denoising step with the host-side commit; returns tokens committed."""
        sh = self.sh
        full = self.full_next and not force_sparse
        tok, conf, ent, E, full_next = self.run(full)
        tok_h = tok.cpu()
        self.full_next = bool(full_next.max().item())
        start = sh.prompt + self.block * sh.block
        committed = 0
        changed = []
        for b in range(sh.B):
            for j in range(sh.block):
                t = int(tok_h[b, j])
                if t >= 0:
                    self.tokens_host[b, start + j] = t
                    self.history[b].append(start + j)
                    changed.append((b, start + j))
                    committed += 1
        if changed:
            rows = torch.full((sh.B, sh.block), -1, dtype=torch.int32)
            cnts = [0] * sh.B
            for b, p in changed:
                rows[b, cnts[b]] = p
                cnts[b] += 1
            self.tokens.copy_(self.tokens_host.to(self.dev))
            B.dllm_embed(self.E, self.tokens, self.H0, rows=rows.to(self.dev))
        blk = self.tokens_host[:, start:start + sh.block]
        if bool((blk != self.mask_id).all()) and self.block + 1 < self.n_blocks:
            self.block += 1
            self._set_block_rows()
        else:
            self._refresh_forced()
        return committed

    def done(self) -> bool:
        return bool((self.tokens_host != self.mask_id).all())

    def prefill(self):
        """Caches of every layer from one full forward over the current tokens."""
        self.run(True)
        torch.cuda.synchronize(self.dev)
        self.full_next = False
