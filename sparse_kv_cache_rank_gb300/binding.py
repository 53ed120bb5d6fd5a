"""Thin torch binding of libdllm.so: the C entry points of include/dllm.h under the
same names, taking torch tensors.  Only argument marshalling happens here (shape
and dtype checks, pointers, the current CUDA stream, workspace tensors); every
step of the refresh runs in the library's kernels.  Nothing falls back to another
implementation: a missing library or a failed call raises.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libdllm.so")

DLLM_F32, DLLM_BF16 = 0, 1
STATUS_TIMEOUT, STATUS_COUNT_CLAMP = 1, 2

_lock = threading.Lock()
_lib = None


class DllmError(RuntimeError):
    pass


class dllm_layer(C.Structure):
    _fields_ = [("w_qkv", C.c_void_p), ("w_o", C.c_void_p), ("w_gu", C.c_void_p),
                ("w_down", C.c_void_p), ("gamma1", C.c_void_p), ("gamma2", C.c_void_p),
                ("rope_inv_freq", C.c_void_p),
                ("d", C.c_int), ("n_q", C.c_int), ("n_kv", C.c_int), ("hd", C.c_int), ("F", C.c_int),
                ("eps", C.c_float), ("rope_theta", C.c_float), ("use_rope", C.c_int),
                ("dtype", C.c_int)]


_SIGS = {
    "dllm_last_error": (C.c_char_p, []),
    "dllm_version": (C.c_int, []),
    "dllm_check_status": (C.c_int, [C.POINTER(C.c_uint), C.c_int]),
    "dllm_proxy_score": (C.c_int, [C.c_void_p] * 5 + [C.c_int] * 5 + [C.c_void_p, C.c_size_t, C.c_void_p]),
    "dllm_proxy_workspace_bytes": (C.c_size_t, [C.c_int] * 5),
    "dllm_kl_drift_workspace_bytes": (C.c_size_t, [C.c_int, C.c_int]),
    "dllm_kl_drift": (C.c_int, [C.c_void_p] * 3 + [C.c_int] * 3 + [C.c_void_p, C.c_size_t, C.c_void_p]),
    "dllm_ce_step": (C.c_int, [C.c_void_p] * 6 + [C.c_int] * 2 + [C.c_float] * 5 + [C.c_int, C.c_float, C.c_void_p]),
    "dllm_polestar_commit": (C.c_int, [C.c_void_p] * 7 + [C.c_int] * 2 + [C.c_float] * 2 + [C.c_void_p]),
    "dllm_spherical_kmeans": (C.c_int, [C.c_void_p] * 4 + [C.c_int] * 5 + [C.c_void_p]),
    "dllm_cluster_residual": (C.c_int, [C.c_void_p] * 5 + [C.c_int] * 4 + [C.c_void_p]),
    "dllm_nvfp4_quantize": (C.c_int, [C.c_void_p, C.c_float, C.c_void_p, C.c_void_p, C.c_long, C.c_int, C.c_void_p]),
    "dllm_nvfp4_dequantize": (C.c_int, [C.c_void_p, C.c_void_p, C.c_float, C.c_void_p, C.c_long, C.c_int, C.c_void_p]),
    "dllm_cluster_select": (C.c_int, [C.c_void_p] * 3 + [C.c_int] + [C.c_void_p] * 2 + [C.c_int] * 4 + [C.c_void_p]),
    "dllm_select_topk": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_float,
                                   C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_void_p]),
    "dllm_layer_rho": (C.c_double, [C.c_int] + [C.c_double] * 5),
    "dllm_layer_budget": (C.c_int, [C.c_double, C.c_int]),
    "dllm_packed_layer_bytes": (C.c_size_t, [C.c_int] * 6),
    "dllm_pack_layer": (C.c_int, [C.c_void_p] * 9 + [C.c_int] * 5 + [C.c_float, C.c_float,
                                                                      C.c_int, C.c_int, C.c_void_p,
                                                                      C.c_size_t,
                                                                      C.POINTER(dllm_layer),
                                                                      C.c_void_p]),
    "dllm_refresh_workspace_bytes": (C.c_size_t, [C.POINTER(dllm_layer), C.c_int, C.c_int, C.c_int]),
    "dllm_sparse_layer_refresh": (C.c_int, [C.POINTER(dllm_layer), C.c_void_p, C.c_void_p,
                                            C.c_void_p, C.c_int, C.c_void_p, C.c_void_p,
                                            C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_int,
                                            C.c_int, C.c_void_p, C.c_size_t, C.c_void_p]),
    "dllm_layer_step_workspace_bytes": (C.c_size_t, [C.POINTER(dllm_layer)] + [C.c_int] * 5),
    "dllm_layer_step": (C.c_int, [C.POINTER(dllm_layer)] + [C.c_void_p] * 6 + [C.c_int] * 2 + [C.c_float]
                        + [C.c_void_p] * 5 + [C.c_int] * 3 + [C.c_void_p, C.c_size_t, C.c_void_p]),
    "dllm_set_pdl": (C.c_int, [C.c_int]),
    "dllm_timer_start": (C.c_int, [C.c_int, C.c_int]),
    "dllm_timer_stop": (C.c_int, [C.POINTER(C.c_double), C.POINTER(C.c_int)]),
    "dllm_launch_count": (C.c_ulonglong, []),
    "dllm_gemm_bf16": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int,
                                 C.c_int, C.c_void_p]),
    "dllm_gemm_plan": (C.c_int, [C.c_int] * 6 + [C.c_void_p]),
    "dllm_attention_workspace_bytes": (C.c_size_t, [C.c_int] * 6),
    "dllm_attention": (C.c_int, [C.c_void_p] * 6 + [C.c_int] * 7 + [C.c_void_p, C.c_size_t, C.c_void_p]),
    "dllm_embed": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_void_p] + [C.c_int] * 5
                   + [C.c_void_p]),
    "dllm_rows_rmsnorm": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.c_void_p, C.c_float, C.c_void_p]
                          + [C.c_int] * 4 + [C.c_void_p]),
    "dllm_check_wait_timeout": (C.c_int, [C.c_void_p, C.c_void_p]),
    "dllm_gather_rows": (C.c_int, [C.c_void_p] * 5 + [C.c_int] * 3 + [C.c_void_p]),
    "dllm_gather_rows_n": (C.c_int, [C.c_int] + [C.c_void_p] * 5 + [C.c_int] * 3 + [C.c_void_p]),
    "dllm_commit_entropy_noalloc": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int,
                                              C.c_float, C.c_float] + [C.c_void_p] * 6),
    "dllm_commit_workspace_bytes": (C.c_size_t, [C.c_int, C.c_int, C.c_int]),
    "dllm_lmhead_workspace_bytes": (C.c_size_t, [C.c_int, C.c_int, C.c_int]),
    "dllm_lmhead_commit": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p] + [C.c_int] * 4 +
                           [C.c_float, C.c_float] + [C.c_void_p] * 6 + [C.c_size_t, C.c_void_p]),
    "dllm_commit_entropy": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int,
                                      C.c_float, C.c_float] + [C.c_void_p] * 6 +
                            [C.c_size_t, C.c_void_p]),
}


def exported_symbols():
    """Names of every entry point the binding expects the library to export."""
    return list(_SIGS)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise DllmError(f"libdllm.so not built ({LIB_PATH}); run __graft_entry__.build()")
            L = C.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
        return _lib


def _check(rc: int, what: str):
    if rc != 0:
        msg = lib().dllm_last_error().decode(errors="replace")
        raise DllmError(f"{what} failed ({rc}): {msg}")


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(device=None):
    return C.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return DLLM_BF16
    if t.dtype == torch.float32:
        return DLLM_F32
    raise DllmError(f"unsupported dtype {t.dtype}")


def _cuda(*ts):
    for t in ts:
        if t is not None:
            if not t.is_cuda:
                raise DllmError("tensors must be on a CUDA device")
            if not t.is_contiguous():
                raise DllmError("tensors must be contiguous")


_ws_cache: dict = {}


def _workspace(nbytes: int, device, tag: str) -> torch.Tensor:
    """Caller-side scratch buffer (the library itself never allocates).  One buffer is kept
    per (entry point, device) and reused by every call that passes no `ws`, so calls that
    are ordered on one stream share it safely; calls of the same entry point that may run
    concurrently (different streams without ordering) must each pass their own `ws`."""
    key = (tag, device.index if device.index is not None else torch.cuda.current_device())
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


# --------------------------------------------------------------------------- status
def check_status(reset: bool = True) -> int:
    st = C.c_uint(0)
    rc = lib().dllm_check_status(C.byref(st), 1 if reset else 0)
    if rc == -5:
        raise DllmError(f"device status 0x{st.value:x}: a kernel wait timed out")
    _check(rc, "dllm_check_status")
    return st.value


def dllm_check_wait_timeout():
    """Runs the library's bounded-wait diagnostic (about one second on the device) and
    returns (threads whose wait gave up, the return code of dllm_check_status after it,
    the status bits); the status word is cleared."""
    dev = torch.cuda.current_device()
    out = torch.zeros(1, dtype=torch.int32, device=dev)
    _check(lib().dllm_check_wait_timeout(_ptr(out), _stream(dev)), "dllm_check_wait_timeout")
    st = C.c_uint(0)
    rc = lib().dllm_check_status(C.byref(st), 1)
    return int(out.item()), rc, st.value


# --------------------------------------------------------------------------- measurement
KERNELS = {"proxy_gemm": 1, "cosine": 2, "select": 3, "gather": 4, "qkv": 5, "attention": 6,
           "oproj": 7, "rmsnorm2": 8, "gateup": 9, "down": 10, "vocab": 11, "gemm": 12,
           "kl_drift": 13, "ce": 14, "polestar": 15, "cluster": 16}


def dllm_timer_start(kernel: str, max_launches: int) -> None:
    _check(lib().dllm_timer_start(KERNELS[kernel], int(max_launches)), "dllm_timer_start")


def dllm_timer_stop():
    """-> (total milliseconds over the timed launches, number of timed launches)."""
    ms, n = C.c_double(0), C.c_int(0)
    _check(lib().dllm_timer_stop(C.byref(ms), C.byref(n)), "dllm_timer_stop")
    return ms.value, n.value


def dllm_launch_count() -> int:
    return int(lib().dllm_launch_count())


def dllm_set_pdl(enable: bool) -> bool:
    """Programmatic dependent launch between the library's kernels (default on)."""
    return bool(lib().dllm_set_pdl(1 if enable else 0))


# --------------------------------------------------------------------------- proxy
def dllm_proxy_score(H, Pt, proxy_cache, proxy_cur=None, drift=None, ws=None):
    """H [B,N,d] (bf16|f32), Pt [r,d] same dtype, proxy_cache [B,N,r] f32 ->
    (proxy_cur [B,N,r] f32, drift [B,N] f32)."""
    B, N, d = H.shape
    r = Pt.shape[0]
    if Pt.shape != (r, d) or Pt.dtype != H.dtype:
        raise DllmError("Pt must be [r, d] with H's dtype")
    if proxy_cur is None:
        proxy_cur = torch.empty((B, N, r), dtype=torch.float32, device=H.device)
    if drift is None:
        drift = torch.empty((B, N), dtype=torch.float32, device=H.device)
    _cuda(H, Pt, proxy_cache, proxy_cur, drift)
    need = int(lib().dllm_proxy_workspace_bytes(B, N, d, r, _dtype_code(H)))
    if ws is None and need > 0:
        ws = _workspace(need, H.device, "proxy")
    _check(lib().dllm_proxy_score(_ptr(H), _ptr(Pt), _ptr(proxy_cache), _ptr(proxy_cur), _ptr(drift),
                                  B, N, d, r, _dtype_code(H), _ptr(ws), 0 if ws is None else ws.numel(),
                                  _stream(H.device)), "dllm_proxy_score")
    return proxy_cur, drift


def dllm_kl_drift(proxy_cur, proxy_cache, drift=None, ws=None):
    """proxy_cur, proxy_cache [B,N,r] f32 -> drift [B,N] f32 = KL of the rows' proxy-attention
    distributions (this step against the cached proxies)."""
    B, N, r = proxy_cur.shape
    if proxy_cache.shape != (B, N, r) or proxy_cur.dtype != torch.float32 or proxy_cache.dtype != torch.float32:
        raise DllmError("proxy_cur and proxy_cache must both be [B, N, r] float32")
    if drift is None:
        drift = torch.empty((B, N), dtype=torch.float32, device=proxy_cur.device)
    _cuda(proxy_cur, proxy_cache, drift)
    need = int(lib().dllm_kl_drift_workspace_bytes(B, N))
    if ws is None:
        ws = _workspace(need, proxy_cur.device, "kl")
    _check(lib().dllm_kl_drift(_ptr(proxy_cur), _ptr(proxy_cache), _ptr(drift), B, N, r, _ptr(ws), ws.numel(),
                               _stream(proxy_cur.device)), "dllm_kl_drift")
    return drift


def dllm_ce_step(conf, seen, undecided, committed, state, early=None, q_l=1e-3, q_v=1e-3, R=1e-2,
                 p_v0=1e-2, z=1.645, h_max=4, c_min=0.9):
    """Confidence extrapolation step: conf [B,M] f32, seen/undecided/committed [B,M] uint8,
    state [B,M,5] f32 (updated in place) -> early [B,M] uint8."""
    B, M = conf.shape
    if state.shape != (B, M, 5) or state.dtype != torch.float32 or conf.dtype != torch.float32:
        raise DllmError("conf [B, M] and state [B, M, 5] must be float32")
    for t in (seen, undecided, committed):
        if t.shape != (B, M) or t.dtype != torch.uint8:
            raise DllmError("seen, undecided, committed must be [B, M] uint8")
    if early is None:
        early = torch.empty((B, M), dtype=torch.uint8, device=conf.device)
    _cuda(conf, seen, undecided, committed, state, early)
    _check(lib().dllm_ce_step(_ptr(conf), _ptr(seen), _ptr(undecided), _ptr(committed), _ptr(state),
                              _ptr(early), B, M, float(q_l), float(q_v), float(R), float(p_v0), float(z),
                              int(h_max), float(c_min), _stream(conf.device)), "dllm_ce_step")
    return early


def dllm_polestar_commit(drift, conf, undecided, suffix, selected, history, commit=None, alpha=1.0, tau_s=0.9):
    """Drift-aware commit: drift, conf [B,M] f32; undecided, suffix, selected [B,M] uint8;
    history [B,M,2] f32 (updated in place) -> commit [B,M] uint8."""
    B, M = drift.shape
    if conf.shape != (B, M) or history.shape != (B, M, 2) or history.dtype != torch.float32:
        raise DllmError("conf [B, M] f32 and history [B, M, 2] f32 expected")
    for t in (undecided, suffix, selected):
        if t.shape != (B, M) or t.dtype != torch.uint8:
            raise DllmError("undecided, suffix, selected must be [B, M] uint8")
    if commit is None:
        commit = torch.empty((B, M), dtype=torch.uint8, device=drift.device)
    _cuda(drift, conf, undecided, suffix, selected, history, commit)
    _check(lib().dllm_polestar_commit(_ptr(drift), _ptr(conf), _ptr(undecided), _ptr(suffix), _ptr(selected),
                                      _ptr(history), _ptr(commit), B, M, float(alpha), float(tau_s),
                                      _stream(drift.device)), "dllm_polestar_commit")
    return commit


def dllm_spherical_kmeans(X, C, iters: int, assign=None, xnorm=None):
    """X [B,N,D] f32, C [B,K,D] f32 (initial; refined in place) -> (assign [B,N] int32, xnorm [B,N] f32)."""
    B, N, D = X.shape
    K = C.shape[1]
    if C.shape != (B, K, D) or X.dtype != torch.float32 or C.dtype != torch.float32:
        raise DllmError("X [B, N, D] and C [B, K, D] must be float32")
    if assign is None:
        assign = torch.empty((B, N), dtype=torch.int32, device=X.device)
    if xnorm is None:
        xnorm = torch.empty((B, N), dtype=torch.float32, device=X.device)
    _cuda(X, C, assign, xnorm)
    _check(lib().dllm_spherical_kmeans(_ptr(X), _ptr(C), _ptr(assign), _ptr(xnorm), B, N, D, K, int(iters),
                                       _stream(X.device)), "dllm_spherical_kmeans")
    return assign, xnorm


def dllm_cluster_residual(X, C, assign, xnorm, R=None):
    B, N, D = X.shape
    K = C.shape[1]
    if R is None:
        R = torch.empty_like(X)
    _cuda(X, C, assign, xnorm, R)
    _check(lib().dllm_cluster_residual(_ptr(X), _ptr(C), _ptr(assign), _ptr(xnorm), _ptr(R), B, N, D, K,
                                       _stream(X.device)), "dllm_cluster_residual")
    return R


def dllm_nvfp4_quantize(R, g: float, codes=None, scales=None):
    """R [rows, D] f32 -> (codes [rows, D/2] uint8, scales [rows, D/16] uint8)."""
    R2 = R.reshape(-1, R.shape[-1])
    rows, D = R2.shape
    if codes is None:
        codes = torch.empty((rows, D // 2), dtype=torch.uint8, device=R.device)
    if scales is None:
        scales = torch.empty((rows, D // 16), dtype=torch.uint8, device=R.device)
    _cuda(R2, codes, scales)
    _check(lib().dllm_nvfp4_quantize(_ptr(R2), float(g), _ptr(codes), _ptr(scales), rows, D, _stream(R.device)),
           "dllm_nvfp4_quantize")
    return codes, scales


def dllm_nvfp4_dequantize(codes, scales, g: float, out=None):
    """codes [rows, D/2] uint8, scales [rows, D/16] uint8 -> out [rows, D] f32."""
    rows, half = codes.shape
    D = half * 2
    if out is None:
        out = torch.empty((rows, D), dtype=torch.float32, device=codes.device)
    _cuda(codes, scales, out)
    _check(lib().dllm_nvfp4_dequantize(_ptr(codes), _ptr(scales), float(g), _ptr(out), rows, D,
                                       _stream(codes.device)), "dllm_nvfp4_dequantize")
    return out


def dllm_cluster_select(C_now, C_prev, assign, kc: int, idx=None, count=None):
    """-> (idx [B,N] int32 ascending member rows of the kc most drifted clusters, -1 padded; count [B])."""
    B, K, D = C_now.shape
    N = assign.shape[1]
    if idx is None:
        idx = torch.empty((B, N), dtype=torch.int32, device=C_now.device)
    if count is None:
        count = torch.empty((B,), dtype=torch.int32, device=C_now.device)
    _cuda(C_now, C_prev, assign, idx, count)
    _check(lib().dllm_cluster_select(_ptr(C_now), _ptr(C_prev), _ptr(assign), int(kc), _ptr(idx), _ptr(count),
                                     B, N, D, K, _stream(C_now.device)), "dllm_cluster_select")
    return idx, count


# --------------------------------------------------------------------------- selection
def dllm_select_topk(drift, forced, k: int, min_drift: float = 1e-6, idx=None, count=None):
    """drift [B,N] f32, forced [B,F] int32 (-1 padded) or None ->
    (idx [B,N] int32 ascending, -1 padded;  count [B] int32)."""
    B, N = drift.shape
    F = 0 if forced is None else forced.shape[1]
    if idx is None:
        idx = torch.empty((B, N), dtype=torch.int32, device=drift.device)
    if count is None:
        count = torch.empty((B,), dtype=torch.int32, device=drift.device)
    _cuda(drift, forced, idx, count)
    _check(lib().dllm_select_topk(_ptr(drift), _ptr(forced), F, int(k), float(min_drift), _ptr(idx),
                                  _ptr(count), B, N, _stream(drift.device)), "dllm_select_topk")
    return idx, count


def dllm_layer_rho(l: int, base=0.05, peak=0.30, centre=16.0, sigma_left=6.0, sigma_right=6.0):
    return float(lib().dllm_layer_rho(int(l), base, peak, centre, sigma_left, sigma_right))


def dllm_layer_budget(rho: float, N: int) -> int:
    return int(lib().dllm_layer_budget(float(rho), int(N)))


# --------------------------------------------------------------------------- layer
class Layer:
    """Packed weights of one layer on the device plus the dllm_layer descriptor."""

    def __init__(self, packed: torch.Tensor, desc: dllm_layer):
        self.packed = packed
        self.desc = desc

    @property
    def dtype(self):
        return torch.bfloat16 if self.desc.dtype == DLLM_BF16 else torch.float32


def dllm_pack_layer(w: dict, n_q: int, n_kv: int, hd: int, eps: float = 1e-5,
                    rope_theta: float = 10000.0, use_rope: bool = True) -> Layer:
    """w: device tensors in nn.Linear layout (w_q, w_k, w_v, w_o, w_g, w_u, w_d, gamma1, gamma2)."""
    keys = ("w_q", "w_k", "w_v", "w_o", "w_g", "w_u", "w_d", "gamma1", "gamma2")
    ts = [w[k].contiguous() for k in keys]
    _cuda(*ts)
    dt = _dtype_code(ts[0])
    if any(t.dtype != ts[0].dtype for t in ts):
        raise DllmError("all weights must share one dtype")
    d = ts[7].shape[0]
    F = ts[4].shape[0]
    nbytes = lib().dllm_packed_layer_bytes(d, n_q, n_kv, hd, F, dt)
    packed = torch.empty(nbytes, dtype=torch.uint8, device=ts[0].device)
    desc = dllm_layer()
    _check(lib().dllm_pack_layer(*[_ptr(t) for t in ts], d, n_q, n_kv, hd, F, float(eps),
                                 float(rope_theta), 1 if use_rope else 0, dt, _ptr(packed), nbytes,
                                 C.byref(desc), _stream(ts[0].device)), "dllm_pack_layer")
    return Layer(packed, desc)


def dllm_refresh_workspace_bytes(layer: Layer, B: int, N: int, k_max: int) -> int:
    return int(lib().dllm_refresh_workspace_bytes(C.byref(layer.desc), B, N, k_max))


def dllm_sparse_layer_refresh(layer: Layer, H_in, idx, count, k_max: int, K_cache, V_cache,
                              H_out_cache, proxy_cache=None, proxy_cur=None, ws=None):
    """Refreshes the cache rows idx[b, :count[b]] in place (K_cache, V_cache,
    H_out_cache, and proxy_cache when given)."""
    B, N, d = H_in.shape
    r = 0 if proxy_cache is None else proxy_cache.shape[-1]
    _cuda(H_in, idx, count, K_cache, V_cache, H_out_cache, proxy_cache, proxy_cur)
    need = dllm_refresh_workspace_bytes(layer, B, N, k_max)
    if ws is None:
        ws = _workspace(need, H_in.device, "refresh")
    _check(lib().dllm_sparse_layer_refresh(C.byref(layer.desc), _ptr(H_in), _ptr(idx), _ptr(count),
                                           int(k_max), _ptr(K_cache), _ptr(V_cache),
                                           _ptr(H_out_cache), _ptr(proxy_cache), _ptr(proxy_cur), r,
                                           B, N, _ptr(ws), ws.numel(), _stream(H_in.device)),
           "dllm_sparse_layer_refresh")
    return K_cache, V_cache, H_out_cache


def dllm_layer_step_workspace_bytes(layer: Layer, B: int, N: int, r: int, F: int, k: int) -> int:
    return int(lib().dllm_layer_step_workspace_bytes(C.byref(layer.desc), B, N, r, F, k))


def dllm_layer_step(layer: Layer, Pt, H_in, proxy_cache, proxy_cur, drift, forced, k: int, idx, count,
                    K_cache, V_cache, H_out_cache, min_drift: float = 1e-6, ws=None):
    """One layer's sparse step (proxy + drift, selection with the forced rows, refresh of
    the selected rows) in one library call; writes proxy_cur, drift, idx, count and the
    refreshed cache rows in place."""
    B, N, d = H_in.shape
    r = proxy_cache.shape[-1]
    F = 0 if forced is None else forced.shape[1]
    _cuda(Pt, H_in, proxy_cache, proxy_cur, drift, forced, idx, count, K_cache, V_cache, H_out_cache)
    need = dllm_layer_step_workspace_bytes(layer, B, N, r, F, k)
    if ws is None:
        ws = _workspace(need, H_in.device, "layer_step")
    _check(lib().dllm_layer_step(C.byref(layer.desc), _ptr(Pt), _ptr(H_in), _ptr(proxy_cache), _ptr(proxy_cur),
                                 _ptr(drift), _ptr(forced), F, int(k), float(min_drift), _ptr(idx), _ptr(count),
                                 _ptr(K_cache), _ptr(V_cache), _ptr(H_out_cache), B, N, r, _ptr(ws), ws.numel(),
                                 _stream(H_in.device)), "dllm_layer_step")
    return idx, count


# --------------------------------------------------------------------------- attention alone
def dllm_attention(Q, K_cache, V_cache, idx, count, k_max: int, A=None, ws=None):
    """Q [B*k_max, n_q*hd], caches [B, N, n_kv, hd] -> A [B*k_max, n_q*hd] (zeros for rows
    that are not live)."""
    Bn, N, n_kv, hd = K_cache.shape
    n_q = Q.shape[1] // hd
    if A is None:
        A = torch.empty_like(Q)
    _cuda(Q, K_cache, V_cache, A, idx, count)
    dt = _dtype_code(Q)
    need = int(lib().dllm_attention_workspace_bytes(Bn, N, int(k_max), n_q, hd, dt))
    if ws is None and need > 0:
        ws = _workspace(need, Q.device, "attention")
    _check(lib().dllm_attention(_ptr(Q), _ptr(K_cache), _ptr(V_cache), _ptr(A), _ptr(idx), _ptr(count),
                                int(k_max), Bn, N, n_q, n_kv, hd, dt, _ptr(ws),
                                0 if ws is None else ws.numel(), _stream(Q.device)), "dllm_attention")
    return A


# --------------------------------------------------------------------------- embedding, final norm
def dllm_embed(E, tokens, H, rows=None):
    """H[b, i] = E[tokens[b, i]] for all i, or for the positions rows[b, :] only."""
    B, N, d = H.shape
    V = E.shape[0]
    R = 0 if rows is None else rows.shape[1]
    _cuda(E, tokens, H, rows)
    _check(lib().dllm_embed(_ptr(E), _ptr(tokens), _ptr(rows), R, _ptr(H), B, N, d, V,
                            _dtype_code(H), _stream(H.device)), "dllm_embed")
    return H


def dllm_rows_rmsnorm(H, rows, gamma, eps: float = 1e-5, out=None):
    """out [B*R, d] = RMSNorm(H[b, rows[b, j]]) * gamma."""
    B, N, d = H.shape
    R = rows.shape[1]
    if out is None:
        out = torch.empty((B * R, d), dtype=H.dtype, device=H.device)
    _cuda(H, rows, gamma, out)
    _check(lib().dllm_rows_rmsnorm(_ptr(H), _ptr(rows), R, _ptr(gamma), float(eps), _ptr(out), B, N,
                                   d, _dtype_code(H), _stream(H.device)), "dllm_rows_rmsnorm")
    return out


def dllm_gather_rows(src, idx, count, k_max: int, dst=None):
    """src [B, N, ...] (any row layout, rows of a multiple of 16 bytes) ->
    dst [B*k_max, ...]: the rows idx[b, :count[b]] packed per sequence, zeros after."""
    Bn, N = src.shape[0], src.shape[1]
    row_bytes = src[0, 0].numel() * src.element_size()
    if dst is None:
        dst = torch.empty((Bn * k_max,) + tuple(src.shape[2:]), dtype=src.dtype, device=src.device)
    if dst.numel() * dst.element_size() < Bn * k_max * row_bytes:
        raise DllmError("dst holds fewer than B*k_max rows")
    _cuda(src, idx, count, dst)
    _check(lib().dllm_gather_rows(_ptr(src), _ptr(idx), _ptr(count), int(k_max), _ptr(dst), Bn, N, row_bytes,
                                  _stream(src.device)), "dllm_gather_rows")
    return dst


def dllm_gather_rows_n(srcs, idx, count, k_max: int, dsts=None):
    """The rows idx[b, :count[b]] of several caches [B, N, ...] sharing one selection,
    packed per sequence in one launch -> list of dst [B*k_max, ...] (zeros after)."""
    srcs = list(srcs)
    if not 1 <= len(srcs) <= 4:
        raise DllmError("between 1 and 4 caches")
    Bn, N = srcs[0].shape[0], srcs[0].shape[1]
    if dsts is None:
        dsts = [torch.empty((Bn * k_max,) + tuple(s.shape[2:]), dtype=s.dtype, device=s.device) for s in srcs]
    rb = []
    for s_, d_ in zip(srcs, dsts):
        if s_.shape[:2] != (Bn, N):
            raise DllmError("the caches must share [B, N]")
        rb.append(s_[0, 0].numel() * s_.element_size())
        if d_.numel() * d_.element_size() < Bn * k_max * rb[-1]:
            raise DllmError("dst holds fewer than B*k_max rows")
    _cuda(*srcs, *dsts, idx, count)
    n = len(srcs)
    src_arr = (C.c_void_p * n)(*[_ptr(t) for t in srcs])
    dst_arr = (C.c_void_p * n)(*[_ptr(t) for t in dsts])
    rb_arr = (C.c_int * n)(*rb)
    _check(lib().dllm_gather_rows_n(n, src_arr, dst_arr, rb_arr, _ptr(idx), _ptr(count), int(k_max), Bn, N,
                                    _stream(srcs[0].device)), "dllm_gather_rows_n")
    return dsts


# --------------------------------------------------------------------------- plain GEMM
def dllm_gemm_bf16(X, W, out=None, splits: int = 0):
    """X [M, K] bf16, W [N_out, K] bf16 -> out [M, N_out] fp32 = X W^T (tensor cores)."""
    M, K = X.shape
    N_out = W.shape[0]
    if W.shape != (N_out, K) or X.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
        raise DllmError("X [M,K] and W [N_out,K] must be bf16")
    if out is None:
        out = torch.empty((M, N_out), dtype=torch.float32, device=X.device)
    _cuda(X, W, out)
    _check(lib().dllm_gemm_bf16(_ptr(X), _ptr(W), _ptr(out), M, N_out, K, int(splits),
                                _stream(X.device)), "dllm_gemm_bf16")
    return out


PLAN_FIELDS = ("BN", "splits", "stages", "tok_tiles", "w_tiles", "xrows", "smem", "ctas_per_sm")


def dllm_gemm_plan(M: int, N_out: int, K: int, splits: int = 0, sms: int = 152, slices: int = 0):
    """The tensor-core GEMM's launch plan for this shape on `sms` SMs (host only, no GPU
    needed) -> dict of PLAN_FIELDS.  slices: 0 the plain GEMM, 1 the proxy projection's
    independent K slices, 2 the proxy projection with its drift in the epilogue."""
    info = (C.c_int32 * 8)()
    _check(lib().dllm_gemm_plan(int(M), int(N_out), int(K), int(splits), int(sms), int(slices), info),
           "dllm_gemm_plan")
    return dict(zip(PLAN_FIELDS, list(info)))


# --------------------------------------------------------------------------- vocab
def dllm_commit_entropy(logits, valid, conf_thresh: float = 0.9, tau: float = 2.0, out=None, ws=None):
    """logits [B,M,V] f32, valid [B,M] uint8 ->
    (token [B,M] int32, conf [B,M], entropy [B,M], max_entropy [B], full_next [B] int32)."""
    B, M, V = logits.shape
    dev = logits.device
    if out is None:
        out = (torch.empty((B, M), dtype=torch.int32, device=dev),
               torch.empty((B, M), dtype=torch.float32, device=dev),
               torch.empty((B, M), dtype=torch.float32, device=dev),
               torch.empty((B,), dtype=torch.float32, device=dev),
               torch.empty((B,), dtype=torch.int32, device=dev))
    tok, conf, ent, E, full = out
    _cuda(logits, valid, *out)
    need = int(lib().dllm_commit_workspace_bytes(B, M, V))
    if ws is None:
        ws = _workspace(need, dev, "commit")
    _check(lib().dllm_commit_entropy(_ptr(logits), _ptr(valid), B, M, V, float(conf_thresh),
                                     float(tau), _ptr(tok), _ptr(conf), _ptr(ent), _ptr(E),
                                     _ptr(full), _ptr(ws), ws.numel(), _stream(dev)),
           "dllm_commit_entropy")
    return out


def dllm_lmhead_commit(X, W_lm, valid, conf_thresh: float = 0.9, tau: float = 2.0, out=None, ws=None):
    """X [B*M, d] bf16 (normalised block rows), W_lm [V, d] bf16, valid [B, M] uint8 ->
    the outputs of dllm_commit_entropy on X W_lm^T, without materialising the logits."""
    B, M = valid.shape
    V, d = W_lm.shape
    if X.shape != (B * M, d) or X.dtype != torch.bfloat16 or W_lm.dtype != torch.bfloat16:
        raise DllmError("X [B*M, d] and W_lm [V, d] must be bf16")
    dev = X.device
    if out is None:
        out = (torch.empty((B, M), dtype=torch.int32, device=dev),
               torch.empty((B, M), dtype=torch.float32, device=dev),
               torch.empty((B, M), dtype=torch.float32, device=dev),
               torch.empty((B,), dtype=torch.float32, device=dev),
               torch.empty((B,), dtype=torch.int32, device=dev))
    tok, conf, ent, E, full = out
    _cuda(X, W_lm, valid, *out)
    need = int(lib().dllm_lmhead_workspace_bytes(B, M, V))
    if ws is None:
        ws = _workspace(need, dev, "lmhead")
    _check(lib().dllm_lmhead_commit(_ptr(X), _ptr(W_lm), _ptr(valid), B, M, V, d, float(conf_thresh),
                                    float(tau), _ptr(tok), _ptr(conf), _ptr(ent), _ptr(E), _ptr(full),
                                    _ptr(ws), ws.numel(), _stream(dev)),
           "dllm_lmhead_commit")
    return out


def dllm_commit_entropy_noalloc(logits, valid, conf_thresh: float = 0.9, tau: float = 2.0, out=None):
    """dllm_commit_entropy for callers that cannot allocate device memory: the library
    keeps the scratch in its own fixed device array (no workspace argument).  The caller
    still provides the output tensors (allocated here when `out` is None)."""
    B, M, V = logits.shape
    dev = logits.device
    if out is None:
        out = (torch.empty((B, M), dtype=torch.int32, device=dev),
               torch.empty((B, M), dtype=torch.float32, device=dev),
               torch.empty((B, M), dtype=torch.float32, device=dev),
               torch.empty((B,), dtype=torch.float32, device=dev),
               torch.empty((B,), dtype=torch.int32, device=dev))
    tok, conf, ent, E, full = out
    _cuda(logits, valid, *out)
    _check(lib().dllm_commit_entropy_noalloc(_ptr(logits), _ptr(valid), B, M, V, float(conf_thresh),
                                             float(tau), _ptr(tok), _ptr(conf), _ptr(ent), _ptr(E),
                                             _ptr(full), _stream(dev)),
           "dllm_commit_entropy_noalloc")
    return out
