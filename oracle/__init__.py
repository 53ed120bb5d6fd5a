"""CPU oracle for the sparse KV-cache refresh step -- TEST INFRASTRUCTURE ONLY.

Only `tests/`, `__graft_entry__.smoke()` and the CPU-baseline leg of `bench.py`
may import this package.  The product library never imports, links or calls it.

`oracle.c` holds the arithmetic (plain loops, fp32 storage, double accumulation);
this module compiles it with gcc on first use and wraps it with ctypes so that
callers pass numpy arrays.  `svd.py` builds the proxy matrix with LAPACK in fp64.
Nothing here shares code with the CUDA library.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

from .svd import proxy_matrix, proxy_singular_values  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into _oracle.so (gcc, -O2, no fast-math, no FMA contraction)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Layer(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in
                ("w_q", "w_k", "w_v", "w_o", "w_g", "w_u", "w_d", "gamma1", "gamma2")] + [
        ("d", C.c_int), ("n_q", C.c_int), ("n_kv", C.c_int), ("hd", C.c_int), ("F", C.c_int),
        ("eps", C.c_float), ("rope_theta", C.c_float), ("use_rope", C.c_int)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = C.CDLL(build())
            _lib.oracle_rho.restype = C.c_double
            _lib.oracle_rho.argtypes = [C.c_int] + [C.c_double] * 5
            _lib.oracle_budget.restype = C.c_int
            _lib.oracle_budget.argtypes = [C.c_double, C.c_int]
            _lib.oracle_max_threads.restype = C.c_int
        return _lib


def set_threads(n: int) -> None:
    lib().oracle_set_threads(int(n))


def max_threads() -> int:
    return int(lib().oracle_max_threads())


def _f32(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


# ---------------------------------------------------------------------------
# proxy + drift
# ---------------------------------------------------------------------------
def proxy_score(H, P, proxy_cache):
    """H [B,N,d], P [d,r], proxy_cache [B,N,r] -> (proxy_cur [B,N,r], drift [B,N])."""
    H, P, pc = _f32(H), _f32(P), _f32(proxy_cache)
    B, N, d = H.shape
    r = P.shape[1]
    assert P.shape == (d, r) and pc.shape == (B, N, r)
    cur = np.empty((B, N, r), np.float32)
    drift = np.empty((B, N), np.float32)
    lib().oracle_proxy_score(_p(H), _p(P), _p(pc), _p(cur), _p(drift), B, N, d, r)
    return cur, drift


def rope_row(x, pos: int, theta: float = 10000.0):
    """One head vector rotated at position pos (rotate-half pairs)."""
    x = np.array(x, dtype=np.float32, copy=True)
    lib().oracle_rope_row(_p(x), x.shape[0], int(pos), C.c_float(theta))
    return x


def cosine_drift(cur, cached):
    cur, cached = _f32(cur), _f32(cached)
    r = cur.shape[-1]
    rows = cur.size // r
    out = np.empty(cur.shape[:-1], np.float32)
    lib().oracle_cosine_drift(_p(cur), _p(cached), _p(out), C.c_long(rows), r)
    return out


# ---------------------------------------------------------------------------
# selection and budget
# ---------------------------------------------------------------------------
def select_topk(drift, forced, k: int, min_drift: float = 1e-6):
    """drift [B,N], forced [B,F] (-1 padded) or None -> (idx [B,N] ascending, -1 padded; count [B])."""
    drift = _f32(drift)
    B, N = drift.shape
    if forced is None or np.size(forced) == 0:
        fo, F = None, 0
    else:
        fo = _i32(forced)
        F = fo.shape[1]
    idx = np.empty((B, N), np.int32)
    cnt = np.empty(B, np.int32)
    lib().oracle_select_topk(_p(drift), _p(fo), F, int(k), C.c_float(min_drift), _p(idx), _p(cnt), B, N)
    return idx, cnt


def rho(l: int, base=0.05, peak=0.30, centre=16.0, sigma_left=6.0, sigma_right=6.0) -> float:
    return float(lib().oracle_rho(int(l), base, peak, centre, sigma_left, sigma_right))


def budget(rho_l: float, N: int) -> int:
    return int(lib().oracle_budget(float(rho_l), int(N)))


# ---------------------------------------------------------------------------
# layer
# ---------------------------------------------------------------------------
class Layer:
    """Keeps fp32 copies of one layer's weights alive and exposes the C struct."""

    def __init__(self, w: dict, n_q: int, n_kv: int, hd: int, eps: float = 1e-5,
                 rope_theta: float = 10000.0, use_rope: bool = True):
        self.arrs = {k: _f32(w[k]) for k in
                     ("w_q", "w_k", "w_v", "w_o", "w_g", "w_u", "w_d", "gamma1", "gamma2")}
        d = self.arrs["gamma1"].shape[0]
        F = self.arrs["w_g"].shape[0]
        assert self.arrs["w_q"].shape == (n_q * hd, d)
        assert self.arrs["w_k"].shape == (n_kv * hd, d) and self.arrs["w_v"].shape == (n_kv * hd, d)
        assert self.arrs["w_o"].shape == (d, n_q * hd)
        assert self.arrs["w_u"].shape == (F, d) and self.arrs["w_d"].shape == (d, F)
        self.d, self.n_q, self.n_kv, self.hd, self.F = d, n_q, n_kv, hd, F
        self.s = _Layer(*[_p(self.arrs[k]) for k in
                          ("w_q", "w_k", "w_v", "w_o", "w_g", "w_u", "w_d", "gamma1", "gamma2")],
                        d, n_q, n_kv, hd, F, eps, rope_theta, 1 if use_rope else 0)

    @property
    def d_kv(self):
        return self.n_kv * self.hd


def layer_full(L: Layer, H):
    """Dense forward over every row -> (K_cache, V_cache, H_out), each fp32."""
    H = _f32(H)
    B, N, d = H.shape
    K = np.empty((B, N, L.d_kv), np.float32)
    V = np.empty((B, N, L.d_kv), np.float32)
    O = np.empty((B, N, d), np.float32)
    lib().oracle_layer_full(C.byref(L.s), _p(H), _p(K), _p(V), _p(O), B, N)
    return K, V, O


def layer_refresh(L: Layer, H, idx, count, K_cache, V_cache, H_out_cache,
                  proxy_cache=None, proxy_cur=None, out_mask=None):
    """Sparse refresh at rows idx[b, :count[b]].  Updates the cache arrays in place
    (they must be C-contiguous float32) and returns them."""
    H = _f32(H)
    B, N, d = H.shape
    idx, count = _i32(idx), _i32(count)
    for a in (K_cache, V_cache, H_out_cache):
        assert a.dtype == np.float32 and a.flags.c_contiguous
    r = 0
    if proxy_cache is not None:
        assert proxy_cache.dtype == np.float32 and proxy_cache.flags.c_contiguous
        proxy_cur = _f32(proxy_cur)
        r = proxy_cache.shape[-1]
    mask = None if out_mask is None else np.ascontiguousarray(out_mask, dtype=np.uint8)
    lib().oracle_layer_refresh(C.byref(L.s), _p(H), _p(idx), _p(count), idx.shape[1],
                               _p(K_cache), _p(V_cache), _p(H_out_cache), _p(proxy_cache),
                               _p(proxy_cur), r, B, N, _p(mask))
    return K_cache, V_cache, H_out_cache


def attention_rows(L: Layer, Q, K_cache, V_cache):
    """Attention outputs [c, n_q*hd] of query rows Q [c, n_q*hd] against one sequence's cache."""
    Q, K_cache, V_cache = _f32(Q), _f32(K_cache), _f32(V_cache)
    c = Q.shape[0]
    N = K_cache.shape[0]
    A = np.empty_like(Q)
    lib().oracle_attention_rows(C.byref(L.s), _p(Q), _p(K_cache), _p(V_cache), N, c, _p(A))
    return A


# ---------------------------------------------------------------------------
# vocabulary
# ---------------------------------------------------------------------------
def lmhead(h, gamma_f, W_lm, eps: float = 1e-5):
    h, gamma_f, W_lm = _f32(h), _f32(gamma_f), _f32(W_lm)
    M, d = h.shape
    V = W_lm.shape[0]
    out = np.empty((M, V), np.float32)
    lib().oracle_lmhead(_p(h), _p(gamma_f), _p(W_lm), M, d, V, C.c_float(eps), _p(out))
    return out


def vocab_stats(logits):
    logits = _f32(logits)
    V = logits.shape[-1]
    rows = logits.size // V
    am = np.empty(logits.shape[:-1], np.int32)
    pm = np.empty(logits.shape[:-1], np.float32)
    H = np.empty(logits.shape[:-1], np.float32)
    lib().oracle_vocab_stats(_p(logits), C.c_long(rows), V, _p(am), _p(pm), _p(H))
    return am, pm, H


def commit_rule(argmax, pmax, entropy, valid, conf_thresh=0.9, tau=2.0):
    argmax, pmax, entropy = _i32(argmax), _f32(pmax), _f32(entropy)
    valid = np.ascontiguousarray(valid, dtype=np.uint8)
    B, M = argmax.shape
    tok = np.empty((B, M), np.int32)
    E = np.empty(B, np.float32)
    full = np.empty(B, np.int32)
    lib().oracle_commit_rule(_p(argmax), _p(pmax), _p(entropy), _p(valid), B, M,
                             C.c_float(conf_thresh), C.c_float(tau), _p(tok), _p(E), _p(full))
    return tok, E, full


def commit_entropy(logits, valid, conf_thresh=0.9, tau=2.0):
    """logits [B,M,V], valid [B,M] -> (token, conf, entropy, max_entropy, full_next)."""
    logits = _f32(logits)
    B, M, V = logits.shape
    valid = np.ascontiguousarray(valid, dtype=np.uint8)
    tok = np.empty((B, M), np.int32)
    conf = np.empty((B, M), np.float32)
    ent = np.empty((B, M), np.float32)
    E = np.empty(B, np.float32)
    full = np.empty(B, np.int32)
    lib().oracle_commit_entropy(_p(logits), _p(valid), B, M, V, C.c_float(conf_thresh),
                                C.c_float(tau), _p(tok), _p(conf), _p(ent), _p(E), _p(full))
    return tok, conf, ent, E, full
