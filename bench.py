#!/usr/bin/env python3
"""Throughput of the sparse KV-cache refresh step on GB300.

One step (the "layer" workload, LLaDA-8B-shaped layer: B=1, N=1024, d=4096,
32 MHA heads x 128, SwiGLU 12288, proxy rank 128, update ratio 16% -> k=164):
    dllm_proxy_score   singular proxy + cosine drift of every row
    dllm_select_topk   top-k drifted rows
    dllm_sparse_layer_refresh   gather/RMSNorm, QKV + rotary + KV scatter, attention
                       over the full cache, O + residual, RMSNorm, SwiGLU, down + scatter
on resident inputs; consecutive steps alternate between two drifted inputs so that
every step selects k rows (a refreshed row's cached proxy is the one it was refreshed
with).  The weights (436 MB) exceed the 129 MB L2, so no L2 flush is needed.

Besides the headline line's keys: the end-to-end leg (host inputs in, refreshed rows
out), the CPU oracle timed on whole steps, the next-row kernels, the 32-layer
LLaDA-8B-shaped and 28-layer Dream-7B-shaped stacks, and the other layer
configurations (tiny fp32, Dream-shaped layer, the 36-point long-context sweep).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
Under torchrun every rank runs an independent replica (weak scaling, no collective on
the data path); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "sparse-refresh denoise steps/s & tokens/s (LLaDA-8B shape); % of roofline"
# dram__bytes_read.sum + dram__bytes_write.sum per launch, LLaDA-8B layer at k = 164
# (profiles/layer_step_llada8b_full.md); to be re-taken whenever these kernels change
NCU_TRAFFIC_BYTES = {"gateup": 205.64e6, "qkv": 106.07e6, "down": 110.29e6, "oproj": 36.32e6,
                     "attention": 18.17e6, "proxy_gemm": 9.47e6, "select": 6.13e6}
UNIT = "steps/s"
DATA = "synthetic (seeded random-init weights N(0,0.02), drift model: 10% rows +N(0,0.5), all +N(0,0.05))"


def layer_config(sh, k, world):
    """The `config` object of a layer workload's line (native and reference arms)."""
    return {"workload": f"{sh.name} B={sh.B} N={sh.N} d={sh.d} heads={sh.n_q}x{sh.hd} F={sh.F} "
                        f"r={sh.r} rho={sh.rho} k={k}",
            "l2": "inputs larger than L2 (436 MB of weights per step)" if sh.d >= 1024 else "small layer",
            "parallelism": f"replicas x{world}"}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-full", action="store_true",
                    help="also time the single-thread oracle points that take more than a minute per step")
    ap.add_argument("--no-stack", action="store_true",
                    help="skip the 32-layer LLaDA-8B-shaped and 28-layer Dream-7B-shaped stacks")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other layer configurations (tiny fp32, Dream-shaped, long context)")
    ap.add_argument("--quick-sweep", action="store_true",
                    help="9 long-context points (batch 1, without 50%%) instead of all 36")
    ap.add_argument("--reference-workload", choices=["llada8b-layer", "tiny-fp32"], default="llada8b-layer",
                    help="workload of the reference arm (the small one only for quick checks)")
    ap.add_argument("--profile-step", action="store_true",
                    help="profiling mode: set up the layer workload, warm up, then run ONE layer "
                         "step inside a cudaProfilerStart/Stop range (for ncu --profile-from-start off); "
                         "prints a short JSON line, no measurement")
    ap.add_argument("--profile-proxy", action="store_true",
                    help="one proxy score with the drift in the projection's epilogue (B=4, N=8192) "
                         "inside a profiler range, for ncu")
    ap.add_argument("--profile-kl", action="store_true",
                    help="profiling mode: ONE KL drift call on the layer workload's proxies inside a "
                         "cudaProfilerStart/Stop range; prints a short JSON line, no measurement")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), float(j.get("bf16_tflops_sustained", j["bf16_tflops"])), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# --------------------------------------------------------------------------- clocks
class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- work model
def _proxy_slices(rows, r, d):
    """K slices of the proxy projection's plan on this device (host-only plan query)."""
    import torch
    from sparse_kv_cache_rank_gb300 import binding as B
    sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 152
    return B.dllm_gemm_plan(rows, r, d, sms=sms, slices=1)["splits"]


def layer_kernel_work(sh, M):
    """Algorithmic bytes and FLOPs of each kernel of one layer step with M refreshed rows
    (weights and caches counted once, bf16 = 2 bytes, fp32 = 4).  Up to N = 4096 the
    selection and the gather of the selected rows are one kernel ("select"); with bf16,
    r <= 128 and no K split the proxy projection computes the drift itself ("proxy_gemm"),
    with a K split the selection kernel does ("select")."""
    B, N, d, r, F = sh.B, sh.N, sh.d, sh.r, sh.F
    dq, dkv = sh.d_q, sh.d_kv
    fold = sh.dtype == "bf16" and M <= 256   # the refresh folds the second RMSNorm up to 256 rows
    sel = (4 * B * N + 4 * B * N + 4 * B, 0)
    gat = (2 * M * d * 2 + 8 * M * r, 0)
    if N <= 4096:
        sel, gat = (sel[0] + gat[0], 0), None
    # bf16 with r <= 128 and no K split (the token tiles fill the GPU): the projection's
    # epilogue computes the drift (reads the cached proxies, writes the new ones and the
    # drift); no separate cosine kernel
    slices = _proxy_slices(B * N, r, d) if sh.dtype == "bf16" and d % 64 == 0 and r % 32 == 0 else 1
    fused = sh.dtype == "bf16" and r <= 128 and r % 32 == 0 and d % 64 == 0 and slices == 1
    # the one-call layer step with bf16 K-slice partials or fp32 proxies (r <= 128,
    # N <= 4096): the selection kernel computes the drift, no cosine kernel
    in_select = (sh.dtype == "f32" or slices > 1) and r <= 128 and N <= 4096
    if in_select:
        sel = (sel[0] + 8 * B * N * r + 4 * B * N, 0)
    work = {
        "proxy_gemm": (2 * B * N * d + 2 * r * d + 4 * B * N * r + ((4 * B * N * r + 4 * B * N) if fused else 0),
                       2 * B * N * d * r),
        "cosine": None if (fused or in_select) else (8 * B * N * r + 4 * B * N, 0),
        "select": sel,
        "gather": gat,
        "qkv": (2 * (dq + 2 * dkv) * d + 2 * M * d + 2 * M * (dq + 2 * dkv), 2 * M * d * (dq + 2 * dkv)),
        "attention": (2 * M * dq * 2 + 2 * B * N * 2 * dkv, 4 * M * N * dq),
        # bf16: the second RMSNorm is folded into the O epilogue (which also writes the
        # bf16 h1 * gamma2 operand and the rows' partial squares) and the gate/up epilogue
        "oproj": (2 * d * dq + 2 * M * dq + 2 * M * d + 4 * M * d + (2 * M * d + M * d // 8 if fold else 0),
                  2 * M * dq * d),
        "rmsnorm2": None if fold else (4 * M * d + 2 * M * d, 0),
        "gateup": (2 * 2 * F * d + 2 * M * d + 2 * M * F, 2 * M * d * 2 * F),
        "down": (2 * d * F + 2 * M * F + 4 * M * d + 2 * M * d, 2 * M * F * d),
    }
    return {k: v for k, v in work.items() if v is not None}


# --------------------------------------------------------------------------- native arm
def _layer_weights(sh, seed, dev):
    """Random-init weights N(0, 0.02) of one layer (nn.Linear layout), packed, and the
    layer's proxy matrix from the one-time set-up."""
    import torch
    from sparse_kv_cache_rank_gb300 import binding as B
    from sparse_kv_cache_rank_gb300.proxy_setup import build_proxy_matrix
    bf = torch.float32 if sh.dtype == "f32" else torch.bfloat16
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)

    def randn(*shape):
        return (torch.randn(shape, generator=gen, device=dev, dtype=torch.float32) * 0.02).to(bf)

    d, dq, dkv, F = sh.d, sh.d_q, sh.d_kv, sh.F
    w = {"w_q": randn(dq, d), "w_k": randn(dkv, d), "w_v": randn(dkv, d), "w_o": randn(d, dq),
         "w_g": randn(F, d), "w_u": randn(F, d), "w_d": randn(d, F),
         "gamma1": torch.ones(d, device=dev, dtype=bf), "gamma2": torch.ones(d, device=dev, dtype=bf)}
    layer = B.dllm_pack_layer(w, sh.n_q, sh.n_kv, sh.hd, eps=sh.eps, rope_theta=sh.rope_theta)
    return w, layer, build_proxy_matrix(w["w_v"], w["gamma1"], sh.r)


class LayerWorkload:
    """One layer's resident state for repeated sparse refresh steps: weights (N(0, 0.02)),
    two drifted inputs that alternate step to step, caches from a full refresh of the
    previous input, and the forced rows (the current block's masked rows and the k_recent
    decoded before them) when the shape has a vocabulary block.  `shared` = (w, layer, Pt)
    of another workload with the same layer shape reuses its weights."""

    def __init__(self, sh, seed, dev, shared=None):
        import torch
        from sparse_kv_cache_rank_gb300 import binding as B
        self.B_ = B
        self.sh = sh
        self.dev = dev
        bf = torch.float32 if sh.dtype == "f32" else torch.bfloat16
        self.w, self.layer, self.Pt = shared if shared is not None else _layer_weights(sh, seed, dev)
        gen = torch.Generator(device=dev)
        gen.manual_seed(seed + 1)

        def randn(*shape, std=1.0):
            return torch.randn(shape, generator=gen, device=dev, dtype=torch.float32) * std

        Bn, N, d = sh.B, sh.N, sh.d
        H_prev = randn(Bn, N, d)
        n_hot = int(round(0.1 * N))

        def drifted(base):
            h = base + randn(Bn, N, d, std=0.05)
            for b in range(Bn):
                rows = torch.randperm(N, generator=gen, device=dev)[:n_hot]
                h[b, rows] += randn(n_hot, d, std=0.5)
            return h.to(bf).contiguous()

        self.H = [drifted(H_prev), None]
        self.H[1] = drifted(self.H[0].float())
        H_prev = H_prev.to(bf).contiguous()
        # caches: a full refresh (every row selected) on the previous step's input
        self.K = torch.empty((Bn, N, sh.n_kv, sh.hd), device=dev, dtype=bf)
        self.V = torch.empty_like(self.K)
        self.O = torch.empty((Bn, N, d), device=dev, dtype=bf)
        idx_all = torch.arange(N, device=dev, dtype=torch.int32).repeat(Bn, 1).contiguous()
        cnt_all = torch.full((Bn,), N, device=dev, dtype=torch.int32)
        ws_full = torch.empty(B.dllm_refresh_workspace_bytes(self.layer, Bn, N, N), device=dev, dtype=torch.uint8)
        B.dllm_sparse_layer_refresh(self.layer, H_prev, idx_all, cnt_all, N, self.K, self.V, self.O, ws=ws_full)
        del ws_full, idx_all, cnt_all
        self.pc = torch.empty((Bn, N, sh.r), device=dev, dtype=torch.float32)
        ones = torch.ones_like(self.pc)
        B.dllm_proxy_score(H_prev, self.Pt, ones, proxy_cur=self.pc, drift=torch.empty((Bn, N), device=dev))
        del ones
        self.cur = torch.empty_like(self.pc)
        self.drift = torch.empty((Bn, N), device=dev, dtype=torch.float32)
        self.idx = torch.empty((Bn, N), device=dev, dtype=torch.int32)
        self.cnt = torch.empty((Bn,), device=dev, dtype=torch.int32)
        self.k = B.dllm_layer_budget(sh.rho, N)
        self.forced = None
        self.k_max = self.k
        if sh.V and sh.k_recent:   # the block after the prompt: 8 decoded + the rest masked
            rows = torch.arange(sh.prompt - sh.k_recent, sh.prompt + sh.block - sh.k_recent,
                                device=dev, dtype=torch.int32)
            self.forced = rows.repeat(Bn, 1).contiguous()
            self.k_max = min(N, self.k + rows.numel())
        need = B.dllm_refresh_workspace_bytes(self.layer, Bn, N, self.k_max)
        self.ws = torch.empty(need, device=dev, dtype=torch.uint8)
        pw = int(B.lib().dllm_proxy_workspace_bytes(Bn, N, d, sh.r, B.DLLM_BF16 if sh.dtype == "bf16" else B.DLLM_F32))
        self.ws_proxy = torch.empty(max(pw, 256), device=dev, dtype=torch.uint8)
        self.ws_step = torch.empty(B.dllm_layer_step_workspace_bytes(self.layer, Bn, N, sh.r,
                                                                     0 if self.forced is None else self.forced.shape[1],
                                                                     self.k),
                                   device=dev, dtype=torch.uint8)
        self.H_prev = H_prev
        self.s = 0
        torch.cuda.synchronize(dev)

    def shared(self):
        return self.w, self.layer, self.Pt

    def caches(self):
        """The state a step reads and writes: (K, V, O, proxy cache, proxy, drift)."""
        return self.K, self.V, self.O, self.pc, self.cur, self.drift

    def step(self, H=None, idx=None, cnt=None, caches=None):
        """One layer step through dllm_layer_step (one library call), on this workload's
        caches or on another set of the same shapes."""
        B = self.B_
        if H is None:
            H = self.H[self.s & 1]
        idx = self.idx if idx is None else idx
        cnt = self.cnt if cnt is None else cnt
        K, V, O, pc, cur, drift = self.caches() if caches is None else caches
        self.s += 1
        B.dllm_layer_step(self.layer, self.Pt, H, pc, cur, drift, self.forced, self.k, idx, cnt, K, V, O,
                          ws=self.ws_step)

    def step_calls(self):
        """The same step as the three calls dllm_proxy_score, dllm_select_topk and
        dllm_sparse_layer_refresh."""
        B = self.B_
        H = self.H[self.s & 1]
        self.s += 1
        B.dllm_proxy_score(H, self.Pt, self.pc, proxy_cur=self.cur, drift=self.drift, ws=self.ws_proxy)
        B.dllm_select_topk(self.drift, self.forced, self.k, idx=self.idx, count=self.cnt)
        B.dllm_sparse_layer_refresh(self.layer, H, self.idx, self.cnt, self.k_max, self.K, self.V, self.O,
                                    self.pc, self.cur, ws=self.ws)


def kernel_breakdown(wl, reps=4):
    """Mean CUDA-event duration of each kernel of the step (ms), each timed over `reps`
    steps on the launch stream (outside the throughput pass)."""
    B = wl.B_
    out = {}
    for name in layer_kernel_work(wl.sh, 1):
        B.dllm_timer_start(name, 2 * reps)
        for _ in range(reps):
            wl.step()
        ms, n = B.dllm_timer_stop()
        if n > 0:
            out[name] = ms / n
    return out


def roofline_of(sh, M, kernel_ms, name, sustained):
    """Roofline entry of kernel `name`: algorithmic bytes / FLOPs of one launch over its
    event-timed duration, against the measured HBM copy or bf16 peak (whichever bounds the
    kernel's work).  sustained: compare a tensor-bound kernel with the sustained bf16 figure
    (a kernel timed inside a long step) instead of the burst one."""
    bw, tc, tc_sus, src = peaks()
    nbytes, flops = layer_kernel_work(sh, M)[name]
    s = kernel_ms[name] / 1e3
    if flops / (tc * 1e12) > nbytes / (bw * 1e9):
        peak = tc_sus if sustained else tc
        r = {"bound": "tensor", "achieved": flops / s / 1e12, "peak": peak, "unit": "TFLOP/s"}
    else:
        r = {"bound": "hbm", "achieved": nbytes / s / 1e9, "peak": bw, "unit": "GB/s"}
    r["frac"] = r["achieved"] / r["peak"]
    r["kernel"] = name
    r["peak_source"] = src + (" (sustained bf16)" if r["bound"] == "tensor" and sustained else "")
    return r


def step_roofline_s(sh, M):
    bw, tc, _, _ = peaks()
    return sum(max(b / (bw * 1e9), f / (tc * 1e12)) for b, f in layer_kernel_work(sh, M).values())


def hold_device(dev, us=500.0):
    """Keeps the device busy for about `us` microseconds (a clock-spinning kernel) so that
    a timed region recorded after it opens with its work already queued: the region then
    holds the device time of its steps, not the host's latency in issuing the first one."""
    import torch
    torch.cuda._sleep(int(us * 1e-6 * 2.1e9))


def native(args):
    import torch
    import torch.distributed as dist
    from sparse_kv_cache_rank_gb300 import binding as B
    from sparse_kv_cache_rank_gb300 import replicas, synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    # replicas: the job is world * B independent sequences; this rank owns a contiguous
    # shard of them (B = 1 each here) and seeds its inputs by the shard's first sequence
    sh = synth.LLADA_LAYER
    first, stop = replicas.shard_sequences(world * sh.B, world, rank)
    assert stop - first == sh.B
    wl = LayerWorkload(sh, 1234 + first, dev)
    for _ in range(max(args.warmup, 3)):
        wl.step()
    torch.cuda.synchronize(dev)
    B.check_status()
    M = int(wl.cnt.sum().item())

    # per-kernel breakdown (outside the timed region)
    work = layer_kernel_work(sh, M)
    per_kernel = kernel_breakdown(wl)
    dominant = max(per_kernel, key=per_kernel.get)

    # timed region
    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize(dev)
    launches0 = B.dllm_launch_count()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    hold_device(dev)
    e0.record()
    for _ in range(args.steps):
        wl.step()
    e1.record()
    torch.cuda.synchronize(dev)
    launches = B.dllm_launch_count() - launches0
    # the dominant kernel's launch duration: CUDA events around each of its launches over
    # a second pass of the same K steps.  An event between two launches ends the
    # programmatic-dependent-launch overlap, so the pass that gives the throughput runs
    # without them.
    B.dllm_timer_start(dominant, args.steps)
    e2 = torch.cuda.Event(enable_timing=True)
    e3 = torch.cuda.Event(enable_timing=True)
    hold_device(dev)
    e2.record()
    for _ in range(args.steps):
        wl.step()
    e3.record()
    torch.cuda.synchronize(dev)
    dom_ms, dom_n = B.dllm_timer_stop()
    barrier()
    clk = clocks.stop()
    elapsed = e0.elapsed_time(e1) / 1e3
    instrumented_ms = e2.elapsed_time(e3) / args.steps
    B.check_status()

    # the same steps as three library calls each (proxy, selection, refresh)
    for _ in range(3):
        wl.step_calls()
    e4 = torch.cuda.Event(enable_timing=True)
    e5 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    hold_device(dev)
    e4.record()
    for _ in range(args.steps):
        wl.step_calls()
    e5.record()
    torch.cuda.synchronize(dev)
    three_calls_ms = e4.elapsed_time(e5) / args.steps
    e2e_elapsed, e2e_bytes = e2e_measure(wl, args.steps, barrier)

    # the job's time is the slowest replica's
    elapsed, e2e_elapsed = replicas.max_over_ranks([elapsed, e2e_elapsed], device=dev)

    roof = roofline_of(sh, M, {dominant: dom_ms / max(dom_n, 1)}, dominant, sustained=False)
    # DRAM bytes (read + write) per launch from the committed ncu capture; None for a
    # kernel not captured there or changed since
    roof["traffic"] = NCU_TRAFFIC_BYTES.get(dominant)
    roof["timing"] = ("CUDA events around each launch of the kernel on its stream, over a second pass "
                      f"of the {args.steps} timed steps ({instrumented_ms * 1e3:.1f} us/step with the events)")
    steps_per_s = world * args.steps / elapsed
    config = layer_config(sh, wl.k, world)
    result = {
        "metric": METRIC, "value": steps_per_s, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": DATA, "config": config,
        "tokens_per_s": steps_per_s * sh.B * sh.N,
        "refreshed_rows_per_s": steps_per_s * M,
        "rows_per_step": M,
        "timing": (f"CUDA events around {args.steps} back-to-back steps on one stream, inputs resident; "
                   "the region opens after a short clock-spinning kernel, so it starts with the steps queued"),
        "roofline": roof,
        "step_roofline_frac": step_roofline_s(sh, M) / (elapsed / args.steps),
        "three_calls_ms_per_step": three_calls_ms,
        "kernel_ms": {k: round(v, 5) for k, v in per_kernel.items()},
        "kernel_roofline": {k: round(roofline_of(sh, M, per_kernel, k, False)["frac"], 4) for k in per_kernel
                            if work[k][0] > 0},
        "e2e": {"value": world * args.steps / e2e_elapsed, "unit": UNIT, **e2e_bytes},
        "gpu_launches": int(launches),
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(sh, args.cpu_full)
    result["next_rows"] = {"kl_drift": kl_drift_measure(wl, args.steps, args.warmup),
                           "confidence_extrapolation": ce_measure(dev, args.steps, args.warmup),
                           "drift_aware_commit": polestar_measure(dev, args.steps, args.warmup),
                           "cluster_proxy": cluster_measure(dev, args.steps, args.warmup)}
    shared = wl.shared()
    del wl
    torch.cuda.empty_cache()
    if not args.no_stack:
        result["stack"] = stack_measure(dev, args.steps, args.warmup)
        torch.cuda.empty_cache()
        result["dream_stack"] = dream_stack_measure(dev, min(args.steps, 20), args.warmup)
        torch.cuda.empty_cache()
    if not args.no_configs:
        result["configs"] = config_points(dev, shared, args.quick_sweep)
    del shared
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


def e2e_batches(n, cap):
    """Batch sizes for n end-to-end steps: 1, 1, 2, 4 ... up to cap at the start and back
    down to 1 at the end, so that the first step waits for one upload only and the last
    read-back is one step's."""
    head = [b for b in (1, 1, 2, 4, 8, 16) if b < cap] + [cap]
    tail = head[::-1]
    if n <= sum(head) + sum(tail):
        return [1] * n
    mid = n - sum(head) - sum(tail)
    return head + [cap] * (mid // cap) + ([mid % cap] if mid % cap else []) + tail


def e2e_measure(wl, steps, barrier, slots=8, batch=4):
    """The same steps through the same calls with host buffers: every step uploads its
    input from pinned host memory and brings its result back -- the refreshed rows of the
    output cache, of the key cache and of the value cache and the selection -- inside the
    timed region.  The steps share one set of caches, as in the device-resident loop.
    Right after each step the compute stream packs that step's refreshed rows (one
    dllm_gather_rows_n launch, before the next step can rewrite them) into the step's
    slot; inputs, selections and packed rows live in `slots` slots used in turn.  A second
    stream does every copy: it uploads each step's input as soon as its slot is free and
    reads back a batch of steps' results once the batch has finished.  The compute stream
    waits on one event (the upload of the batch's last input) and records one per batch
    of up to `batch` steps (each such wait ends the programmatic-launch overlap between two
    steps' kernels); the batches grow from 1 to `batch` steps at the start and shrink back
    at the end (e2e_batches).  -> (seconds for `steps` steps, byte counts per step)."""
    import torch
    B = wl.B_
    dev = wl.dev
    sh = wl.sh
    km = wl.k_max
    Hh = [wl.H[i & 1].cpu().pin_memory() for i in range(slots)]   # step parity = slot parity
    Hd = [torch.empty_like(wl.H[0]) for _ in range(slots)]
    idx_d = [torch.empty_like(wl.idx) for _ in range(slots)]
    cnt_d = [torch.empty_like(wl.cnt) for _ in range(slots)]
    rows_d = [[torch.empty((sh.B * km,) + tuple(t.shape[2:]), dtype=t.dtype, device=dev) for t in (wl.O, wl.K, wl.V)]
              for _ in range(slots)]
    idx_h = [torch.empty(wl.idx.shape, dtype=torch.int32).pin_memory() for _ in range(slots)]
    cnt_h = [torch.empty(wl.cnt.shape, dtype=torch.int32).pin_memory() for _ in range(slots)]
    rows_h = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in rows_d[0]] for _ in range(slots)]
    main = torch.cuda.current_stream(dev)
    cs = torch.cuda.Stream(dev)
    ready = [torch.cuda.Event() for _ in range(slots)]   # the input of the step in a slot is resident
    read_back = torch.cuda.Event()

    def upload(s):   # on the copy stream
        sl = s % slots
        Hd[sl].copy_(Hh[sl], non_blocking=True)
        ready[sl].record(cs)

    def read_result(s):   # on the copy stream
        sl = s % slots
        idx_h[sl].copy_(idx_d[sl], non_blocking=True)
        cnt_h[sl].copy_(cnt_d[sl], non_blocking=True)
        for dsrc, hdst in zip(rows_d[sl], rows_h[sl]):
            hdst.copy_(dsrc, non_blocking=True)

    def e2e_steps(n, start_event=None):
        sizes = e2e_batches(n, batch)
        with torch.cuda.stream(cs):
            if start_event is not None:
                cs.wait_event(start_event)
            for s in range(min(slots, n)):
                upload(s)
        first = 0
        for bs in sizes:
            last = first + bs - 1
            main.wait_event(ready[last % slots])   # uploads complete in order
            for s in range(first, last + 1):
                sl = s % slots
                wl.step(Hd[sl], idx=idx_d[sl], cnt=cnt_d[sl])
                B.dllm_gather_rows_n((wl.O, wl.K, wl.V), idx_d[sl], cnt_d[sl], km, rows_d[sl])
            done = torch.cuda.Event()
            done.record(main)
            with torch.cuda.stream(cs):   # this batch's results out, then the inputs of its slots' next steps
                cs.wait_event(done)
                for s in range(first, last + 1):
                    read_result(s)
                for s in range(first + slots, min(last + slots + 1, n)):
                    upload(s)
            first = last + 1
        read_back.record(cs)
        main.wait_event(read_back)
        return n

    e2e_steps(2 * slots)
    torch.cuda.synchronize(dev)
    barrier()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    f0.record()
    e2e_steps(steps, f0)
    f1.record()
    torch.cuda.synchronize(dev)
    barrier()
    # the rows read back are the refreshed ones: compare the last step's packed output rows
    # with the device cache (a consistency check of the copies, not of the method)
    sl = (steps - 1) % slots
    c = int(cnt_h[sl][0])
    got = rows_h[sl][0][:c].to(dev)
    want = wl.O[0, idx_h[sl][0, :c].to(dev).long()]
    if not torch.equal(got, want):
        raise RuntimeError("e2e read-back does not match the refreshed rows")
    d2h = idx_h[0].numel() * 4 + cnt_h[0].numel() * 4 + sum(t.numel() * t.element_size() for t in rows_h[0])
    return f0.elapsed_time(f1) / 1e3, {"h2d_bytes_per_step": int(Hh[0].numel() * Hh[0].element_size()),
                                       "d2h_bytes_per_step": int(d2h),
                                       "d2h": "refreshed rows of the output, key and value caches "
                                              f"({sh.B}x{km} rows each, packed by dllm_gather_rows_n right "
                                              "after the step) + the selection",
                                       "copies": f"{slots} input/result slots; one event wait per batch of "
                                                 f"steps: {e2e_batches(steps, batch)}"}


# --------------------------------------------------------------------------- full stack
def stale_proxies(st, seed):
    """Cached proxies of every layer taken from a drifted copy of the layer's current
    input -- the drift model of the layer workloads (+N(0, 0.05) on every row, +N(0, 0.5)
    on 10% of the rows) applied at every depth, the state a layer's cache reaches when its
    inputs moved since it last refreshed them.  Restoring them before a partial step makes
    every layer score drift on every row, so each refreshes its full budget rho(l)."""
    import torch
    from sparse_kv_cache_rank_gb300 import binding as B
    dev = st.dev
    sh = st.sh
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    out = torch.empty_like(st.pc_all)
    ones = torch.ones_like(st.pc_all[0])
    drift = torch.empty((sh.B, sh.N), device=dev)
    n_hot = int(round(0.1 * sh.N))
    H = st.H0
    for l, L in enumerate(st.layers):
        X = H.float() + torch.randn(H.shape, generator=gen, device=dev) * 0.05
        for b in range(sh.B):
            rows = torch.randperm(sh.N, generator=gen, device=dev)[:n_hot]
            X[b, rows] += torch.randn((n_hot, sh.d), generator=gen, device=dev) * 0.5
        B.dllm_proxy_score(X.to(H.dtype).contiguous(), L.Pt, ones, proxy_cur=out[l], drift=drift)
        H = L.O
    torch.cuda.synchronize(dev)
    return out


def _second_block(st, seed):
    """The state at the start of the second generation block: the first block decoded
    (random ids), its last k_recent positions the recent history, so the forced rows are
    the new block's masked positions plus the k_recent recent ones."""
    import torch
    from sparse_kv_cache_rank_gb300 import binding as B
    sh = st.sh
    g = torch.Generator()
    g.manual_seed(seed)
    start = sh.prompt
    st.tokens_host[:, start:start + sh.block] = torch.randint(0, sh.V - 1, (sh.B, sh.block), generator=g,
                                                              dtype=torch.int32)
    for h in st.history:
        h.clear()
        h.extend(range(start + sh.block - st.k_recent, start + sh.block))
    st.tokens.copy_(st.tokens_host.to(st.dev))
    B.dllm_embed(st.E, st.tokens, st.H0)
    st.block = 1
    st._set_block_rows()


def _stack_forced_sparse(st, steps, warmup, seed):
    """The partial denoising step at every layer's budget (see stale_proxies), timed from
    replays of one captured CUDA graph (restore of the cached proxies + the step) and, for
    comparison, issued eagerly through the binding."""
    import torch
    pc_stale = stale_proxies(st, seed)

    def step():
        st.pc_all.copy_(pc_stale)
        return st.forward(False)

    st.pc_all.copy_(pc_stale)
    rec = []
    st.forward(False, record=rec)
    rows = [int(r["cnt"].sum().item()) for r in rec]
    g = st.graph(step, warmup=max(warmup, 2))
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize(st.dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        g.replay()
    e1.record()
    torch.cuda.synchronize(st.dev)
    dt = e0.elapsed_time(e1) / 1e3 / steps
    committed = int((st.out[0] >= 0).sum().item())
    # the same step issued call by call from the host (no graph)
    t0 = time.perf_counter()
    e0.record()
    for _ in range(steps):
        step()
    t_issue = (time.perf_counter() - t0) / steps
    e1.record()
    torch.cuda.synchronize(st.dev)
    dt_eager = e0.elapsed_time(e1) / 1e3 / steps
    del g
    return dt, dt_eager, t_issue, committed, rows


def _decode_loop(st, warmup, decode_steps):
    """Rule-driven decoding from a fresh prefill, each step replayed from the stack's
    captured graphs, with the host-side commit (one device->host read per step)."""
    import torch
    st.capture()
    st.prefill()
    for _ in range(max(warmup, 2)):
        st.decode_step()
    torch.cuda.synchronize(st.dev)
    n_full, toks = 0, 0
    t0 = time.perf_counter()
    for _ in range(decode_steps):
        n_full += 1 if st.full_next else 0
        toks += st.decode_step()
    torch.cuda.synchronize(st.dev)
    return time.perf_counter() - t0, n_full, toks


def stack_measure(dev, steps, warmup, decode_steps=48):
    """32-layer LLaDA-8B-shaped stack (N=768: 512 prompt + 256 generation, block 32,
    vocab 126464, rho(l) piecewise Gaussian, 8 recent tokens forced).

    forced_sparse: the denoising step with the full/partial decision overridden to
      partial, every layer at its budget rho(l) plus the forced rows (cached proxies from
      the drift model at every depth, restored inside each timed step), device-timed from
      CUDA graph replays; the same step issued eagerly is reported beside it.
    rule_driven: the decode loop with the host-side commit (one device->host read per
      step), wall-clock timed; with random weights the maximum entropy always exceeds
      tau, so every step is a full forward.
    """
    import torch
    from sparse_kv_cache_rank_gb300 import synth
    from sparse_kv_cache_rank_gb300.stack import DecodeStack
    sh = synth.LLADA_STACK
    t0 = time.perf_counter()
    st = DecodeStack(sh, 4321, dev, k_recent=8)
    _second_block(st, 5)
    st.prefill()
    setup_s = time.perf_counter() - t0
    dt, dt_eager, t_issue, committed, rows = _stack_forced_sparse(st, steps, warmup, 99)
    forced = int((st.forced >= 0).sum().item())
    dec_s, n_full, toks = _decode_loop(st, warmup, decode_steps)
    res = {
        "workload": f"llada8b-stack layers={sh.layers} B={sh.B} N={sh.N} d={sh.d} V={sh.V} "
                    f"rho(l)=0.05+0.25exp(-(l-16)^2/72) k_recent=8",
        "forced_sparse": {"steps_per_s": 1.0 / dt, "ms_per_step": dt * 1e3,
                          "tokens_per_s": committed / dt, "context_tokens_per_s": sh.B * sh.N / dt,
                          "rows_refreshed_per_layer": rows, "budget_per_layer": st.budgets,
                          "forced_rows": forced,
                          "eager": {"ms_per_step": dt_eager * 1e3, "host_issue_ms_per_step": t_issue * 1e3},
                          "timing": "cuda events around CUDA graph replays of the step (the cached-proxy "
                                    "restore included)"},
        "rule_driven": {"steps": decode_steps, "warmup": max(warmup, 2), "steps_per_s": decode_steps / dec_s,
                        "tokens_per_s": toks / dec_s, "full_steps": n_full,
                        "timing": "wall clock, graph-replayed steps incl. one device->host read and the "
                                  "host commit per step"},
        "setup_s": setup_s,
    }
    del st
    torch.cuda.empty_cache()
    return res


def dream_stack_measure(dev, steps, warmup, decode_steps=8):
    """28-layer Dream-7B-shaped stack (Qwen2.5-7B layout: d=3584, 28 query / 4 KV heads x
    128, FFN 18944), batch 8, N=2048 (1024 prompt + 1024 generation, block 32), vocab
    152064, uniform 16 % update ratio (k = 328 per sequence) plus the block's rows and the
    8 most recent tokens forced; the same two modes as the LLaDA stack."""
    import torch
    from sparse_kv_cache_rank_gb300 import synth
    from sparse_kv_cache_rank_gb300.stack import DecodeStack
    sh = synth.DREAM_STACK
    t0 = time.perf_counter()
    st = DecodeStack(sh, 2468, dev, uniform_rho=sh.rho, k_recent=8)
    _second_block(st, 5)
    st.prefill()
    setup_s = time.perf_counter() - t0
    dt, dt_eager, t_issue, committed, rows = _stack_forced_sparse(st, steps, warmup, 98)
    forced = int((st.forced >= 0).sum().item())
    dec_s, n_full, toks = _decode_loop(st, 2, decode_steps)
    res = {"workload": f"dream7b-stack layers={sh.layers} B={sh.B} N={sh.N} d={sh.d} "
                       f"heads={sh.n_q}q/{sh.n_kv}kv x {sh.hd} F={sh.F} V={sh.V} rho={sh.rho} k_recent=8",
           "forced_sparse": {"steps_per_s": 1.0 / dt, "ms_per_step": dt * 1e3,
                             "context_tokens_per_s": sh.B * sh.N / dt, "committed_tokens_per_s": committed / dt,
                             "rows_refreshed_per_layer": rows, "budget_per_layer": st.budgets[0],
                             "forced_rows": forced,
                             "eager": {"ms_per_step": dt_eager * 1e3, "host_issue_ms_per_step": t_issue * 1e3},
                             "steps": steps,
                             "timing": "cuda events around CUDA graph replays of the step (the cached-proxy "
                                       "restore included)"},
           "rule_driven": {"steps": decode_steps, "warmup": 2, "steps_per_s": decode_steps / dec_s,
                           "tokens_per_s": toks / dec_s, "full_steps": n_full,
                           "timing": "wall clock, graph-replayed steps incl. one device->host read and the "
                                     "host commit per step"},
           "setup_s": setup_s}
    del st
    torch.cuda.empty_cache()
    return res


def layer_point(sh, dev, steps, warmup, seed=77, shared=None):
    """Layer-steps/s of one configuration (CUDA events over `steps` resident steps), the
    per-kernel event times and the dominant kernel's roofline fraction."""
    import torch
    wl = LayerWorkload(sh, seed, dev, shared=shared)
    for _ in range(max(warmup, 3)):
        wl.step()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    hold_device(dev)
    e0.record()
    for _ in range(steps):
        wl.step()
    e1.record()
    torch.cuda.synchronize(dev)
    dt = e0.elapsed_time(e1) / 1e3 / steps
    rows = int(wl.cnt.sum().item())
    per_kernel = kernel_breakdown(wl, reps=3)
    res = {"B": sh.B, "N": sh.N, "rho": sh.rho, "rows_per_step": rows, "dtype": sh.dtype,
           "steps_per_s": 1.0 / dt, "ms_per_step": dt * 1e3, "tokens_per_s": sh.B * sh.N / dt,
           "refreshed_rows_per_s": rows / dt}
    if sh.dtype != "bf16":   # fp32 on the CUDA cores: per-kernel times, no bf16 roofline
        res["kernel_ms"] = {k: round(v, 5) for k, v in per_kernel.items()}
    else:
        dom = max(per_kernel, key=per_kernel.get)
        res["kernel_ms"] = {k: round(v, 5) for k, v in per_kernel.items()}
        res["roofline"] = roofline_of(sh, rows, per_kernel, dom, sustained=True)
        res["kernel_roofline"] = {k: round(roofline_of(sh, rows, per_kernel, k, True)["frac"], 4)
                                  for k in per_kernel if layer_kernel_work(sh, rows)[k][0] > 0}
        res["step_roofline_frac"] = step_roofline_s(sh, rows) / dt
    del wl
    torch.cuda.empty_cache()
    return res


GRAPH_TIMING = ("a CUDA graph of back-to-back calls (the library's launches, captured once), "
                "CUDA events around its replays, outside the timed region")


def _graph_time(call, steps, warmup, dev):
    """Seconds per call: `steps` calls captured in a CUDA graph, replayed after warm-up, so
    the host's per-call cost does not hide the device time of small kernels."""
    import torch
    for _ in range(max(warmup, 3)):
        call()
    torch.cuda.synchronize(dev)
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for _ in range(steps):
            call()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(3):
        g.replay()
    e1.record()
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / 1e3 / (3 * steps)


# fp32 FMA rate of the GPU: 152 SMs x 128 fp32 lanes x 2 FLOP x 2.07 GHz (maximum SM clock)
FP32_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def kl_drift_measure(wl, steps, warmup):
    """The attention-distribution drift (KL of proxy-attention rows, this step against the
    cached proxies) on the layer's proxies: B x N x N x r scores for each of the two steps,
    fp32 on the CUDA cores.  CUDA events around `steps` back-to-back launches."""
    import torch
    B_ = wl.B_
    Bn, N, r = wl.cur.shape
    out = torch.empty((Bn, N), dtype=torch.float32, device=wl.dev)
    s = _graph_time(lambda: B_.dllm_kl_drift(wl.cur, wl.pc, out), steps, warmup, wl.dev)
    flops = 2 * 2 * Bn * N * N * r          # two score products of 2 N^2 r FLOP each
    achieved = flops / s / 1e12
    return {"workload": f"B={Bn} N={N} r={r}", "us_per_launch": s * 1e6, "flop": flops,
            "roofline": {"bound": "alu", "achieved": achieved, "peak": FP32_PEAK_TFLOPS,
                         "unit": "TFLOP/s", "frac": achieved / FP32_PEAK_TFLOPS,
                         "peak_source": "fp32 FMA lanes x maximum SM clock"},
            "timing": GRAPH_TIMING}


def ce_measure(dev, steps, warmup):
    """Confidence extrapolation step (Kalman predict + update of every token's confidence
    state and the early-commit decision) on the LLaDA block (B = 1, M = 32) and on 64
    sequences x 1024 positions; CUDA events around back-to-back launches."""
    import torch
    from sparse_kv_cache_rank_gb300 import binding as B_
    out = {}
    for name, (Bn, M) in {"block": (1, 32), "wide": (64, 1024)}.items():
        gen = torch.Generator(device=dev)
        gen.manual_seed(7)
        conf = torch.rand((Bn, M), generator=gen, device=dev)
        state = torch.zeros((Bn, M, 5), device=dev)
        ones = torch.ones((Bn, M), dtype=torch.uint8, device=dev)
        committed = (torch.rand((Bn, M), generator=gen, device=dev) < 0.5).to(torch.uint8)
        early = torch.empty((Bn, M), dtype=torch.uint8, device=dev)
        B_.dllm_ce_step(conf, torch.zeros_like(ones), ones, committed, state, early)
        s = _graph_time(lambda: B_.dllm_ce_step(conf, ones, ones, committed, state, early), steps, warmup, dev)
        nbytes = Bn * M * (4 + 3 + 2 * 20 + 1)   # conf, flags, state in and out, decision
        out[name] = {"workload": f"B={Bn} M={M}", "us_per_launch": s * 1e6, "bytes": nbytes,
                     "gb_per_s": nbytes / s / 1e9,
                     "note": "latency-bound at these sizes (one CTA per sequence, O(M) work)",
                     "timing": GRAPH_TIMING}
    return out


def polestar_measure(dev, steps, warmup):
    """Drift-aware commit (drift delta against each token's drift history, dynamic threshold,
    suffix rule) over the 256 generated positions of the LLaDA stack (B = 1) and over
    64 x 1024 tokens."""
    import torch
    from sparse_kv_cache_rank_gb300 import binding as B_
    out = {}
    for name, (Bn, M) in {"generation": (1, 256), "wide": (64, 1024)}.items():
        gen = torch.Generator(device=dev)
        gen.manual_seed(11)
        drift = torch.rand((Bn, M), generator=gen, device=dev)
        conf = torch.rand((Bn, M), generator=gen, device=dev)
        ones = torch.ones((Bn, M), dtype=torch.uint8, device=dev)
        suffix = torch.zeros_like(ones)
        suffix[:, 32:] = 1
        sel = (torch.rand((Bn, M), generator=gen, device=dev) < 0.3).to(torch.uint8)
        hist = torch.zeros((Bn, M, 2), device=dev)
        commit = torch.empty_like(ones)
        s = _graph_time(lambda: B_.dllm_polestar_commit(drift, conf, ones, suffix, sel, hist, commit),
                        steps, warmup, dev)
        nbytes = Bn * M * (4 + 4 + 3 + 2 * 8 + 1)
        out[name] = {"workload": f"B={Bn} M={M}", "us_per_launch": s * 1e6, "bytes": nbytes,
                     "gb_per_s": nbytes / s / 1e9, "note": "elementwise, latency-bound at these sizes",
                     "timing": GRAPH_TIMING}
    return out


def cluster_measure(dev, steps, warmup):
    """Cluster-granular proxy over a local window of the LLaDA stack (prefix, current and
    suffix blocks: 96 rows x d = 4096 hidden states, K = 16 clusters, 4 Lloyd rounds): k-means,
    residuals, NVFP4 quantisation of the residuals, selection of the 4 most drifted
    clusters' rows."""
    import torch
    from sparse_kv_cache_rank_gb300 import binding as B_
    Bn, N, D, K = 1, 96, 4096, 16
    gen = torch.Generator(device=dev)
    gen.manual_seed(5)
    X = torch.randn((Bn, N, D), generator=gen, device=dev)
    C0 = X[:, :K].clone()
    C = C0.clone()
    Cprev = C0.clone()
    assign = torch.empty((Bn, N), dtype=torch.int32, device=dev)
    xnorm = torch.empty((Bn, N), device=dev)
    R = torch.empty_like(X)
    codes = torch.empty((Bn * N, D // 2), dtype=torch.uint8, device=dev)
    scales = torch.empty((Bn * N, D // 16), dtype=torch.uint8, device=dev)
    idx = torch.empty((Bn, N), dtype=torch.int32, device=dev)
    cnt = torch.empty((Bn,), dtype=torch.int32, device=dev)

    def pipeline():
        C.copy_(C0)
        B_.dllm_spherical_kmeans(X, C, 4, assign, xnorm)
        B_.dllm_cluster_residual(X, C, assign, xnorm, R)
        B_.dllm_nvfp4_quantize(R, 1e-3, codes, scales)
        B_.dllm_cluster_select(C, Cprev, assign, 4, idx, cnt)

    s = _graph_time(pipeline, steps, warmup, dev)
    nbytes = Bn * N * D * 4
    return {"workload": f"B={Bn} window={N} rows d={D} K={K} iters=4 kc=4", "us_per_step": s * 1e6,
            "launches_per_step": 2 * 4 + 2 + 3, "window_bytes": nbytes,
            "compressed_bytes": Bn * N * (D // 2 + D // 16),
            "note": "launch-bound at a 96-row window (13 small launches)", "timing": GRAPH_TIMING}


def config_points(dev, shared, quick):
    """The other layer configurations: the tiny fp32 layer (forced block rows), the
    Dream-7B-shaped layer (batch 8, GQA) and the long-context sweep of the LLaDA-8B-shaped
    layer, N x batch x update ratio (all 36 points; quick: batch 1 without 50 %), every
    bf16 point with its per-kernel times and the dominant kernel's roofline fraction.  The
    sweep points share the layer's weights with the headline workload."""
    import dataclasses
    from sparse_kv_cache_rank_gb300 import synth
    out = {"tiny_fp32": layer_point(synth.TINY, dev, 100, 5)}
    dream = dataclasses.replace(synth.DREAM_STACK, name="dream7b-layer", layers=1, V=0)
    out["dream7b_layer"] = layer_point(dream, dev, 20, 3)
    pts = []
    for sh in synth.sweep_shapes():
        if quick and (sh.B != 1 or sh.rho == 0.5):
            continue
        pts.append(layer_point(sh, dev, 10 if sh.B * sh.N * sh.rho > 20000 else 20, 3, shared=shared))
    out["long_context"] = pts
    return out


# --------------------------------------------------------------------------- oracle legs
def cpu_model() -> str:
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for line in r.stdout.splitlines():
            if line.split(":")[0].strip() == "Model name":
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.processor() or platform.machine()


class OracleLayer:
    """One layer's state on the host for whole oracle steps: fp32 copies of the weights,
    the proxy matrix, the two alternating inputs, the caches and cached proxies, the
    forced rows.  Each step is the native step's work: the proxy and drift of all B*N
    rows, the selection, the refresh of the selected rows (caches updated in place)."""

    def __init__(self, orc, sh, w, P, H, K, V, O, pc, forced):
        self.orc, self.sh = orc, sh
        self.L = orc.Layer(w, sh.n_q, sh.n_kv, sh.hd, eps=sh.eps, rope_theta=sh.rope_theta)
        self.P, self.H, self.forced = P, H, forced
        self.state0 = (K, V, O, pc)
        self.reset()

    def reset(self):
        """Back to the first step's state: caches and cached proxies of the previous input."""
        self.K, self.V, self.O, self.pc = (a.copy() for a in self.state0)
        self.s = 0

    def step(self, k):
        orc, sh = self.orc, self.sh
        H = self.H[self.s & 1]
        self.s += 1
        cur, drift = orc.proxy_score(H, self.P, self.pc)
        idx, cnt = orc.select_topk(drift, self.forced, k)
        orc.layer_refresh(self.L, H, idx, cnt, self.K, self.V, self.O, self.pc, cur)
        return int(cnt.sum())


def _time_oracle(ol, k, threads, budget_s, max_reps=8):
    """Whole oracle steps at `threads` threads: one step, then more while the total stays
    within budget_s.  -> (seconds per step, steps timed, rows per step)."""
    ol.orc.set_threads(threads)
    ol.reset()
    t0 = time.perf_counter()
    rows = ol.step(k)
    t1 = time.perf_counter() - t0
    reps = 1
    tot = t1
    while reps < max_reps and tot + t1 <= budget_s:
        t0 = time.perf_counter()
        ol.step(k)
        tot += time.perf_counter() - t0
        reps += 1
    return tot / reps, reps, rows


def cpu_baseline(sh, full):
    """The oracle, as it stands, timed on the host cores: whole layer steps (no sample is
    scaled up) from the first step's state, each with all host threads and with one
    thread, for the LLaDA-8B-shaped layer at its 16 % budget and at 100 % (the full
    recompute) and for the tiny fp32 layer.  The inputs are drawn on the host with the
    native workload's shapes, distributions and construction (reference_inputs).  Points
    whose single-thread step would exceed a minute (from the all-thread time x the thread
    count) are listed as not run unless `full`."""
    import oracle as orc
    from sparse_kv_cache_rank_gb300 import synth
    orc.build()
    cores = os.cpu_count() or 1
    orc.set_threads(cores)
    pts = []
    ol = reference_inputs(orc, sh, 1234)
    ot = reference_inputs(orc, synth.TINY, 77)
    k = orc.budget(sh.rho, sh.N)
    cases = [("llada8b-layer", ol, k), ("llada8b-layer 100%", ol, sh.N),
             ("tiny-fp32", ot, orc.budget(synth.TINY.rho, synth.TINY.N)), ("tiny-fp32 100%", ot, synth.TINY.N)]
    head = None
    for name, o, k in cases:
        t_all, reps, rows = _time_oracle(o, k, cores, 20.0)
        pts.append({"point": name, "threads": cores, "s_per_step": t_all, "steps_per_s": 1.0 / t_all,
                    "steps_timed": reps, "rows_per_step": rows})
        if name == "llada8b-layer":
            head = (t_all, reps, rows)
        if full or t_all * cores <= 60.0:
            t1, reps1, _ = _time_oracle(o, k, 1, 60.0)
            pts.append({"point": name, "threads": 1, "s_per_step": t1, "steps_per_s": 1.0 / t1,
                        "steps_timed": reps1, "rows_per_step": rows})
        else:
            pts.append({"point": name, "threads": 1, "not_run": "cap: one step > 60 s expected "
                        f"({t_all * cores:.0f} s from the {cores}-thread time); run with --cpu-full"})
    t_all, reps, rows = head
    return {"value": 1.0 / t_all, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{reps} whole LLaDA-8B-shaped layer steps (proxy of all {sh.N} rows, selection, refresh "
                      f"of {rows} rows) from the first step's state, on host-drawn inputs of the same workload, "
                      f"{cores} threads; not extrapolated",
            "cpu_model": cpu_model(), "points": pts}


def reference_inputs(orc, sh, seed):
    """The native arm's workload drawn on the host (same shapes, distributions and
    construction: N(0, 0.02) weights, the SVD proxy, two drifted inputs, caches from the
    oracle's dense forward on the previous input, cached proxies of that input)."""
    from sparse_kv_cache_rank_gb300 import synth
    w = synth.layer_weights(sh, seed)
    P = synth.round_bf16(orc.proxy_matrix(w["w_v"], w["gamma1"], sh.r).astype(np.float32)) \
        if sh.dtype == "bf16" else orc.proxy_matrix(w["w_v"], w["gamma1"], sh.r).astype(np.float32)
    H_prev, H0, _ = synth.hidden_pair(sh, seed + 1)
    H1 = synth.drifted(sh, H0, seed + 2)
    L = orc.Layer(w, sh.n_q, sh.n_kv, sh.hd, eps=sh.eps, rope_theta=sh.rope_theta)
    rnd = synth.round_bf16 if sh.dtype == "bf16" else (lambda a: a)
    K, V, O = (rnd(a) for a in orc.layer_full(L, H_prev))
    pc, _ = orc.proxy_score(H_prev, P, np.ones((sh.B, sh.N, sh.r), np.float32))
    forced = None
    if sh.V and sh.k_recent:
        rows = np.arange(sh.prompt - sh.k_recent, sh.prompt + sh.block - sh.k_recent, dtype=np.int32)
        forced = np.repeat(rows[None], sh.B, 0)
    del L
    return OracleLayer(orc, sh, w, P, [H0, H1], K, V, O, pc, forced)


def reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle as orc
    from sparse_kv_cache_rank_gb300 import synth
    orc.build()
    cores = os.cpu_count() or 1
    orc.set_threads(cores)
    sh = synth.TINY if args.reference_workload == "tiny-fp32" else synth.LLADA_LAYER
    ol = reference_inputs(orc, sh, 1234)
    k = orc.budget(sh.rho, sh.N)
    for _ in range(args.warmup):
        ol.step(k)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        ol.step(k)
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    v = 1.0 / dt
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 / v, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": DATA, "config": layer_config(sh, k, args.gpus),
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{args.steps} whole layer steps of the CPU oracle (proxy of all rows, "
                                   f"selection, refresh of the selected rows) after {args.warmup} warm-up "
                                   f"steps, {cores} threads",
                         "cpu_model": cpu_model()},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def profile_step(args):
    """One warmed-up layer step inside a profiler range: the launches an external
    profiler captures are exactly those of one timed bench step."""
    import torch
    from sparse_kv_cache_rank_gb300 import binding as B
    from sparse_kv_cache_rank_gb300 import synth
    dev = torch.device("cuda", 0)
    wl = LayerWorkload(synth.LLADA_LAYER, 1234, dev)
    for _ in range(max(args.warmup, 3)):
        wl.step()
    torch.cuda.synchronize(dev)
    torch.cuda.profiler.start()
    wl.step()
    torch.cuda.synchronize(dev)
    torch.cuda.profiler.stop()
    B.check_status()
    print(json.dumps({"profile_step": "llada8b-layer", "rows": int(wl.cnt.sum())}), flush=True)


def profile_kl(args):
    """One warmed-up KL drift call on the layer step's proxies inside a profiler range."""
    import torch
    from sparse_kv_cache_rank_gb300 import binding as B
    from sparse_kv_cache_rank_gb300 import synth
    dev = torch.device("cuda", 0)
    wl = LayerWorkload(synth.LLADA_LAYER, 1234, dev)
    for _ in range(max(args.warmup, 3)):
        wl.step()
    out = torch.empty(wl.drift.shape, dtype=torch.float32, device=dev)
    for _ in range(3):
        B.dllm_kl_drift(wl.cur, wl.pc, out)
    torch.cuda.synchronize(dev)
    torch.cuda.profiler.start()
    B.dllm_kl_drift(wl.cur, wl.pc, out)
    torch.cuda.synchronize(dev)
    torch.cuda.profiler.stop()
    B.check_status()
    print(json.dumps({"profile_kl": "llada8b-layer proxies", "N": int(wl.cur.shape[1])}), flush=True)


def profile_proxy(args):
    """One warmed-up proxy score of the long-context batch (B = 4, N = 8192, d = 4096,
    r = 128: the projection needs no K split and computes the drift in its epilogue)
    inside a profiler range."""
    import torch
    from sparse_kv_cache_rank_gb300 import binding as B
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(11)
    Bn, N, d, r = 4, 8192, 4096, 128
    H = torch.randn((Bn, N, d), generator=gen, device=dev).to(torch.bfloat16)
    Pt = (torch.randn((r, d), generator=gen, device=dev) * 0.02).to(torch.bfloat16)
    pc = torch.randn((Bn, N, r), generator=gen, device=dev)
    cur = torch.empty_like(pc)
    drift = torch.empty((Bn, N), device=dev)
    for _ in range(3):
        B.dllm_proxy_score(H, Pt, pc, proxy_cur=cur, drift=drift)
    torch.cuda.synchronize(dev)
    torch.cuda.profiler.start()
    B.dllm_proxy_score(H, Pt, pc, proxy_cur=cur, drift=drift)
    torch.cuda.synchronize(dev)
    torch.cuda.profiler.stop()
    B.check_status()
    print(json.dumps({"profile_proxy": f"B={Bn} N={N} d={d} r={r}"}), flush=True)


def main():
    args = parse()
    if args.profile_step:
        profile_step(args)
    elif args.profile_proxy:
        profile_proxy(args)
    elif args.profile_kl:
        profile_kl(args)
    elif args.impl == "reference":
        reference(args)
    else:
        native(args)


if __name__ == "__main__":
    main()
