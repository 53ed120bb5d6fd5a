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
does every step of the computation (library kernels).  Weights are random N(0, 0.02)
from a seeded generator (no trained checkpoint exists here).
"""
from __future__ import annotations

import dataclasses
import math
from collections import deque

import torch

from . import binding as B
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
    def __init__(self, shape: LayerShape, seed: int, device, rho: RhoSchedule | None = None,
                 uniform_rho: float | None = None, k_recent: int = 8, conf_thresh: float = 0.9,
                 tau: float = 2.0, proxy_method: str = "lowrank", keep_weights: bool = False,
                 keep_logits: bool = False):
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
        self.layers = []
        self.weights = [] if keep_weights else None
        self.keep_logits = keep_logits   # materialise the block's logits (else the fused LM head)
        self.logits = None
        for _ in range(sh.layers):
            w = {"w_q": randn(dq, d, std=0.02), "w_k": randn(dkv, d, std=0.02),
                 "w_v": randn(dkv, d, std=0.02), "w_o": randn(d, dq, std=0.02),
                 "w_g": randn(F, d, std=0.02), "w_u": randn(F, d, std=0.02), "w_d": randn(d, F, std=0.02),
                 "gamma1": torch.ones(d, device=device, dtype=bf),
                 "gamma2": torch.ones(d, device=device, dtype=bf)}
            layer = B.dllm_pack_layer(w, sh.n_q, sh.n_kv, sh.hd, eps=sh.eps, rope_theta=sh.rope_theta)
            Pt = B.build_proxy_matrix(w["w_v"], w["gamma1"], sh.r, method=proxy_method, generator=gen)
            if keep_weights:
                self.weights.append(w)
            del w
            K = torch.empty((Bn, N, sh.n_kv, sh.hd), device=device, dtype=bf)
            self.layers.append(_Layer(layer, Pt, K, torch.empty_like(K),
                                      torch.empty((Bn, N, d), device=device, dtype=bf),
                                      torch.zeros((Bn, N, sh.r), device=device, dtype=torch.float32),
                                      torch.zeros((Bn, N, sh.r), device=device, dtype=torch.float32)))
        self.E = randn(sh.V, d, std=0.02)
        self.W_lm = randn(sh.V, d, std=0.02)
        self.gamma_f = torch.ones(d, device=device, dtype=bf)
        self.mask_id = sh.V - 1
        # tokens: prompt ids uniform in [0, V-2], generation region masked
        self.tokens = torch.full((Bn, N), self.mask_id, dtype=torch.int32, device=device)
        self.tokens[:, :sh.prompt] = torch.randint(0, sh.V - 1, (Bn, sh.prompt), generator=gen,
                                                   device=device, dtype=torch.int32)
        self.H0 = torch.empty((Bn, N, d), device=device, dtype=bf)
        B.dllm_embed(self.E, self.tokens, self.H0)
        self.tokens_host = self.tokens.cpu()
        self.block = 0
        self.history = [deque(maxlen=k_recent) for _ in range(Bn)]
        self.full_next = True
        # scratch
        self.drift = torch.empty((Bn, N), device=device, dtype=torch.float32)
        self.idx = torch.empty((Bn, N), device=device, dtype=torch.int32)
        self.cnt = torch.empty((Bn,), device=device, dtype=torch.int32)
        self.idx_all = torch.arange(N, device=device, dtype=torch.int32).repeat(Bn, 1).contiguous()
        self.cnt_all = torch.full((Bn,), N, device=device, dtype=torch.int32)
        self.ones = torch.ones((Bn, N, sh.r), device=device, dtype=torch.float32)
        ws = max(B.dllm_refresh_workspace_bytes(L.layer, Bn, N, N) for L in self.layers[:1])
        self.ws = torch.empty(ws, device=device, dtype=torch.uint8)
        self.budgets = [self.budget(l) for l in range(sh.layers)]
        self.rows_refreshed = [0] * sh.layers
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
        self.block_rows = pos.repeat(sh.B, 1).to(self.dev).contiguous()
        self._refresh_forced()

    def _refresh_forced(self):
        """Masked positions of the current block plus the k most recently decoded ones."""
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
        self.forced = torch.tensor(rows, dtype=torch.int32).to(self.dev)
        self.valid = torch.stack(valid).to(self.dev).contiguous()

    # ------------------------------------------------------------------ device step
    def forward(self, full: bool, H0=None):
        """Layers + LM head + commit.  Returns device tensors (token, conf, entropy, E, full_next)."""
        sh = self.sh
        H = self.H0 if H0 is None else H0
        F = self.forced.shape[1]
        for l, L in enumerate(self.layers):
            B.dllm_proxy_score(H, L.Pt, L.pc, proxy_cur=L.cur, drift=self.drift)
            if full:
                B.dllm_sparse_layer_refresh(L.layer, H, self.idx_all, self.cnt_all, sh.N, L.K, L.V, L.O,
                                            L.pc, L.cur, ws=self.ws)
            else:
                k = self.budgets[l]
                B.dllm_select_topk(self.drift, self.forced, k, idx=self.idx, count=self.cnt)
                B.dllm_sparse_layer_refresh(L.layer, H, self.idx, self.cnt, min(sh.N, k + F), L.K, L.V,
                                            L.O, L.pc, L.cur, ws=self.ws)
            H = L.O
        X = B.dllm_rows_rmsnorm(H, self.block_rows, self.gamma_f, sh.eps)
        if self.keep_logits:
            logits = B.dllm_gemm_bf16(X, self.W_lm).view(sh.B, sh.block, sh.V)
            self.logits = logits
            return B.dllm_commit_entropy(logits, self.valid, self.conf_thresh, self.tau)
        # LM head fused with the softmax statistics (the logits are never stored)
        return B.dllm_lmhead_commit(X, self.W_lm, self.valid, self.conf_thresh, self.tau)

    def count_rows(self, full: bool):
        """Rows refreshed per layer by one step (synchronises; for reporting)."""
        sh = self.sh
        H = self.H0
        F = self.forced.shape[1]
        out = []
        for l, L in enumerate(self.layers):
            if full:
                out.append(sh.B * sh.N)
            else:
                B.dllm_proxy_score(H, L.Pt, L.pc, proxy_cur=L.cur, drift=self.drift)
                B.dllm_select_topk(self.drift, self.forced, self.budgets[l], idx=self.idx, count=self.cnt)
                out.append(int(self.cnt.sum().item()))
                B.dllm_sparse_layer_refresh(L.layer, H, self.idx, self.cnt, min(sh.N, self.budgets[l] + F),
                                            L.K, L.V, L.O, L.pc, L.cur, ws=self.ws)
            H = L.O
        return out

    # ------------------------------------------------------------------ decode loop
    def decode_step(self, force_sparse: bool = False):
        """One denoising step with the host-side commit; returns tokens committed."""
        sh = self.sh
        full = self.full_next and not force_sparse
        tok, conf, ent, E, full_next = self.forward(full)
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
        self.forward(True)
        torch.cuda.synchronize(self.dev)
        self.full_next = False
