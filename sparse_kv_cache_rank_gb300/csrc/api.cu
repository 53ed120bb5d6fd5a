// api.cu -- the extern "C" entry points of libdllm.so (declared in include/dllm.h):
// argument checks, workspace carving and the launch sequence of each call.
#include <nvtx3/nvToolsExt.h>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"

#define DLLM_EXPORT extern "C" __attribute__((visibility("default")))

namespace dllm {

// Device status word (DLLM_STATUS_* bits); kernels receive its device address.
__device__ unsigned g_status_word;

namespace {

thread_local std::string t_err;

int fail(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_err = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char *what) {
    return fail(DLLM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define CHECK_ARG(cond, ...)                                   \
    do {                                                       \
        if (!(cond)) return fail(DLLM_ERR_INVALID_ARG, __VA_ARGS__); \
    } while (0)

#define CHECK_CUDA(expr, what)                   \
    do {                                         \
        cudaError_t e_ = (expr);                 \
        if (e_ != cudaSuccess) return cuda_fail(e_, what); \
    } while (0)

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned8(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Refreshed rows (B * k_max) up to which the bf16 refresh folds the second RMSNorm into
// the O and gate/up epilogues (measured: a launch saved at the 164-row LLaDA-8B step; at
// 2624 rows of the Dream-7B-shaped layer the heavier epilogues cost more than the norm).
constexpr int kFoldNormRows = 256;

size_t el_size(int dtype) { return dtype == DLLM_BF16 ? 2 : 4; }

cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

constexpr int kMaxDev = 64;

unsigned *status_ptr() {
    static unsigned *ptrs[kMaxDev] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<unsigned *>(p);
    }
    return ptrs[dev];
}


// ---------------------------------------------------------------- measurement support
std::atomic<unsigned long long> g_launches{0};

struct KernelTimer {
    std::mutex mu;
    int armed = 0;
    int cap = 0, n = 0;
    std::vector<cudaEvent_t> ev;
} g_timer;

// NVTX range names of the kernels (DLLM_KERNEL_* ids): a profiler shows each library
// launch inside "dllm:<kernel>" (nvtx3 is header-only; without a tool attached the calls
// return at once).
const char *kernel_range_name(int id) {
    static const char *names[] = {"dllm:other",     "dllm:proxy_gemm", "dllm:cosine",  "dllm:select",
                                  "dllm:gather",    "dllm:qkv",        "dllm:attention", "dllm:oproj",
                                  "dllm:rmsnorm2",  "dllm:gateup",     "dllm:down",    "dllm:vocab",
                                  "dllm:gemm",      "dllm:kl_drift",   "dllm:ce",      "dllm:polestar",
                                  "dllm:cluster"};
    return id > 0 && id < (int)(sizeof(names) / sizeof(names[0])) ? names[id] : names[0];
}

// Counts the launches of one library call site, opens an NVTX range named after the
// kernel around them and, when the timer is armed for this kernel, brackets them with a
// pair of events on the launch stream.
struct Launch {
    cudaEvent_t stop = nullptr;
    cudaStream_t st;
    Launch(int kernel_id, cudaStream_t s, int nlaunch = 1) : st(s) {
        g_launches.fetch_add((unsigned long long)nlaunch, std::memory_order_relaxed);
        nvtxRangePushA(kernel_range_name(kernel_id));
        if (g_timer.armed != kernel_id) return;
        std::lock_guard<std::mutex> lock(g_timer.mu);
        if (g_timer.armed != kernel_id || g_timer.n >= g_timer.cap) return;
        cudaEvent_t start = g_timer.ev[2 * g_timer.n];
        stop = g_timer.ev[2 * g_timer.n + 1];
        ++g_timer.n;
        cudaEventRecord(start, st);
    }
    ~Launch() {
        if (stop) cudaEventRecord(stop, st);
        nvtxRangePop();
    }
};

struct PackLayout {
    size_t qkv, o, gu, down, g1, g2, freq, total;
};

PackLayout pack_layout(int d, int n_q, int n_kv, int hd, int F, int dtype) {
    const size_t el = el_size(dtype);
    PackLayout L{};
    size_t off = 0;
    L.qkv = off;
    off = align256(off + (size_t)(n_q + 2 * n_kv) * hd * d * el);
    L.o = off;
    off = align256(off + (size_t)d * n_q * hd * el);
    L.gu = off;
    off = align256(off + (size_t)2 * F * d * el);
    L.down = off;
    off = align256(off + (size_t)d * F * el);
    L.g1 = off;
    off = align256(off + (size_t)d * el);
    L.g2 = off;
    off = align256(off + (size_t)d * el);
    L.freq = off;
    off = align256(off + (size_t)(hd / 2) * 4);
    L.total = off;
    return L;
}

struct RefreshWs {
    size_t xn, q, a, h1, xn2, u, rope, ss, total;
};

RefreshWs refresh_ws(const dllm_layer *W, int B, int N, int k_max) {
    const size_t M = (size_t)B * k_max, el = el_size(W->dtype);
    const size_t dq = (size_t)W->n_q * W->hd;
    RefreshWs r{};
    size_t off = 0;
    r.xn = off;
    off = align256(off + M * W->d * el);
    r.q = off;
    off = align256(off + M * dq * el);
    r.a = off;
    off = align256(off + M * dq * el);
    r.h1 = off;
    off = align256(off + M * W->d * 4);
    r.xn2 = off;
    off = align256(off + M * W->d * el);
    r.u = off;
    off = align256(off + M * W->F * el);
    r.rope = off;
    off = align256(off + M * (size_t)(W->hd / 2) * sizeof(float2));
    r.ss = off;   // partial squares of h1 per 32 features (the folded second RMSNorm)
    off = align256(off + M * (size_t)(W->d / 32) * 4);
    (void)N;
    r.total = off + 256;   // room to align the caller's base
    return r;
}

int check_layer(const dllm_layer *W) {
    CHECK_ARG(W, "layer is NULL");
    CHECK_ARG(W->dtype == DLLM_BF16 || W->dtype == DLLM_F32, "dtype must be DLLM_BF16 or DLLM_F32");
    CHECK_ARG(W->d > 0 && W->n_q > 0 && W->n_kv > 0 && W->F > 0, "layer sizes must be positive");
    if (W->hd != 64 && W->hd != 128) return fail(DLLM_ERR_UNSUPPORTED, "hd must be 64 or 128 (got %d)", W->hd);
    CHECK_ARG(W->n_q % W->n_kv == 0, "n_q must be a multiple of n_kv");
    CHECK_ARG(W->w_qkv && W->w_o && W->w_gu && W->w_down && W->gamma1 && W->gamma2,
              "layer weight pointer is NULL");
    if (W->dtype == DLLM_BF16) {
        if (W->d % 64 || W->F % 64 || (W->n_q * W->hd) % 64)
            return fail(DLLM_ERR_UNSUPPORTED, "bf16 path needs d, F, n_q*hd multiples of 64");
    } else {
        if (W->d % 32 || W->F % 16)
            return fail(DLLM_ERR_UNSUPPORTED, "f32 path needs d % 32 == 0 and F % 16 == 0");
    }
    return DLLM_OK;
}

}  // namespace

int num_sms() {
    static int cache[kMaxDev] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 148;
    if (!cache[dev]) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = n > 0 ? n : 148;
    }
    return cache[dev];
}

}  // namespace dllm

using namespace dllm;

DLLM_EXPORT const char *dllm_last_error(void) { return t_err.c_str(); }

DLLM_EXPORT int dllm_version(void) { return 113; }

DLLM_EXPORT int dllm_check_status(unsigned *status_out, int reset) {
    CHECK_CUDA(cudaDeviceSynchronize(), "cudaDeviceSynchronize");
    unsigned v = 0;
    CHECK_CUDA(cudaMemcpyFromSymbol(&v, g_status_word, sizeof v), "cudaMemcpyFromSymbol");
    if (reset) {
        const unsigned z = 0;
        CHECK_CUDA(cudaMemcpyToSymbol(g_status_word, &z, sizeof z), "cudaMemcpyToSymbol");
    }
    if (status_out) *status_out = v;
    if (v & DLLM_STATUS_TIMEOUT) return fail(DLLM_ERR_TIMEOUT, "a kernel wait timed out (status 0x%x)", v);
    if (v & DLLM_STATUS_SMEM_LAYOUT)
        return fail(DLLM_ERR_CUDA, "a GEMM found its shared memory misaligned and skipped its work (status 0x%x)", v);
    return DLLM_OK;
}

DLLM_EXPORT int dllm_check_wait_timeout(int32_t *gave_up, void *stream) {
    CHECK_ARG(gave_up, "null pointer");
    CHECK_CUDA(wait_timeout_check(gave_up, status_ptr(), as_stream(stream)), "wait check launch");
    return DLLM_OK;
}

// ------------------------------------------------------------------ proxy score
namespace {
// bf16 with r <= 128 and no K split (the token tiles fill the GPU): the projection
// computes the drift in its epilogue.  Otherwise independent K slices write fp32 partials
// (or one slice its proxies) that the cosine kernel sums in order.
bool proxy_fused(int B, int N, int d, int r, int dtype) {
    return dtype == DLLM_BF16 && gemm_tc_cosine_ok(B * N, r, d);
}

int proxy_slices(int B, int N, int d, int r, int dtype) {
    if (dtype != DLLM_BF16 || B <= 0 || N <= 0 || d % 64 || r % 32) return 1;
    return gemm_tc_slices_count(B * N, r, d);
}
}  // namespace

DLLM_EXPORT size_t dllm_proxy_workspace_bytes(int B, int N, int d, int r, int dtype) {
    if (B <= 0 || N <= 0 || d <= 0 || r <= 0 || (long long)B * N > INT_MAX) return 0;
    const int s = proxy_slices(B, N, d, r, dtype);
    return s > 1 ? (size_t)s * B * N * r * sizeof(float) + 256 : 0;
}

DLLM_EXPORT int dllm_proxy_score(const void *H, const void *Pt, const float *proxy_cache,
                                 float *proxy_cur, float *drift, int B, int N, int d, int r,
                                 int dtype, void *ws, size_t ws_bytes, void *stream) {
    CHECK_ARG(H && Pt && proxy_cache && proxy_cur && drift, "null pointer");
    CHECK_ARG(B > 0 && N > 0 && d > 0 && r > 0, "sizes must be positive (B=%d N=%d d=%d r=%d)", B, N, d, r);
    CHECK_ARG((long long)B * N <= INT_MAX, "B*N must fit in an int");
    CHECK_ARG(r <= 1024, "r must be <= 1024");
    CHECK_ARG(aligned16(H) && aligned16(Pt) && aligned16(proxy_cache) && aligned16(proxy_cur),
              "arrays must be 16-byte aligned");
    CHECK_ARG(dtype == DLLM_BF16 || dtype == DLLM_F32, "dtype must be DLLM_BF16 or DLLM_F32");
    if (r % 32) return fail(DLLM_ERR_UNSUPPORTED, "r must be a multiple of 32 (got %d)", r);
    cudaStream_t st = as_stream(stream);
    const int rows = B * N;
    cudaError_t e;
    const int nparts = proxy_slices(B, N, d, r, dtype);
    float *parts = proxy_cur;
    if (nparts > 1) {   // K slices write fp32 partials; the cosine kernel sums them in order
        const size_t need = dllm_proxy_workspace_bytes(B, N, d, r, dtype);
        if (!ws || ws_bytes < need)
            return fail(DLLM_ERR_WORKSPACE, "workspace holds %zu bytes, %zu needed", ws_bytes, need);
        parts = reinterpret_cast<float *>((reinterpret_cast<uintptr_t>(ws) + 255) & ~uintptr_t(255));
    }
    if (dtype == DLLM_BF16 && d % 64) return fail(DLLM_ERR_UNSUPPORTED, "bf16 path needs d % 64 == 0 (got %d)", d);
    if (proxy_fused(B, N, d, r, dtype)) {
        Launch t(DLLM_KERNEL_PROXY_GEMM, st);
        CHECK_CUDA(gemm_tc_cosine(static_cast<const bf16 *>(Pt), r, d, static_cast<const bf16 *>(H), rows,
                                  proxy_cur, proxy_cache, drift, true, status_ptr(), st),
                   "proxy projection launch");
        return DLLM_OK;
    }
    if (dtype == DLLM_BF16) {
        Launch t(DLLM_KERNEL_PROXY_GEMM, st);
        e = gemm_tc_slices(static_cast<const bf16 *>(Pt), r, d, static_cast<const bf16 *>(H), rows, parts,
                           true, status_ptr(), st);
    } else {
        Launch t(DLLM_KERNEL_PROXY_GEMM, st);
        EpiStoreF32 epi{SelRows{}, proxy_cur, r, r};
        e = gemm_simt(static_cast<const float *>(Pt), r, d, static_cast<const float *>(H), rows, epi, st);
    }
    CHECK_CUDA(e, "proxy projection launch");
    {
        Launch t(DLLM_KERNEL_COSINE, st);
        CHECK_CUDA(cosine_drift(parts, nparts, proxy_cache, proxy_cur, drift, rows, r, st),
                   "cosine drift launch");
    }
    return DLLM_OK;
}

DLLM_EXPORT size_t dllm_kl_drift_workspace_bytes(int B, int N) { return kl_drift_workspace_bytes(B, N); }

DLLM_EXPORT int dllm_kl_drift(const float *proxy_cur, const float *proxy_cache, float *drift, int B,
                              int N, int r, void *ws, size_t ws_bytes, void *stream) {
    CHECK_ARG(proxy_cur && proxy_cache && drift, "null pointer");
    CHECK_ARG(B > 0 && N > 0 && r > 0, "sizes must be positive (B=%d N=%d r=%d)", B, N, r);
    CHECK_ARG(B <= 65535, "B must be <= 65535");
    if (r % 32 || r > 256) return fail(DLLM_ERR_UNSUPPORTED, "r must be a multiple of 32 up to 256 (got %d)", r);
    const size_t need = kl_drift_workspace_bytes(B, N);
    if (!ws || ws_bytes < need)
        return fail(DLLM_ERR_WORKSPACE, "workspace holds %zu bytes, %zu needed", ws_bytes, need);
    cudaStream_t st = as_stream(stream);
    Launch t(DLLM_KERNEL_KL_DRIFT, st, 2);
    CHECK_CUDA(kl_drift(proxy_cur, proxy_cache, drift, B, N, r, ws, st), "KL drift launch");
    return DLLM_OK;
}

DLLM_EXPORT int dllm_ce_step(const float *conf, const uint8_t *seen, const uint8_t *undecided,
                             const uint8_t *committed, float *state, uint8_t *early, int B, int M,
                             float q_l, float q_v, float R, float p_v0, float z, int h_max, float c_min,
                             void *stream) {
    CHECK_ARG(conf && seen && undecided && committed && state && early, "null pointer");
    CHECK_ARG(B > 0 && M > 0, "sizes must be positive (B=%d M=%d)", B, M);
    CHECK_ARG(M <= 1024, "M must be <= 1024 (got %d)", M);
    CHECK_ARG(q_l >= 0.f && q_v >= 0.f && R > 0.f && p_v0 >= 0.f && z >= 0.f, "noise levels must be >= 0, R > 0");
    CHECK_ARG(h_max >= 0 && h_max <= 1024, "h_max must be in [0, 1024]");
    cudaStream_t st = as_stream(stream);
    Launch t(DLLM_KERNEL_CE, st);
    const CEParams p{q_l, q_v, R, p_v0, z, c_min, h_max};
    CHECK_CUDA(ce_step(conf, seen, undecided, committed, state, early, B, M, p, st), "CE step launch");
    return DLLM_OK;
}

DLLM_EXPORT int dllm_polestar_commit(const float *drift, const float *conf, const uint8_t *undecided,
                                     const uint8_t *suffix, const uint8_t *selected, float *history,
                                     uint8_t *commit, int B, int M, float alpha, float tau_s, void *stream) {
    CHECK_ARG(drift && conf && undecided && suffix && selected && history && commit, "null pointer");
    CHECK_ARG(B > 0 && M > 0, "sizes must be positive (B=%d M=%d)", B, M);
    CHECK_ARG(aligned8(history), "history must be 8-byte aligned");
    CHECK_ARG(alpha >= 0.f, "alpha must be >= 0");
    cudaStream_t st = as_stream(stream);
    Launch t(DLLM_KERNEL_POLESTAR, st);
    CHECK_CUDA(polestar_commit(drift, conf, undecided, suffix, selected, history, commit, (long)B * M, alpha,
                               tau_s, st),
               "drift-aware commit launch");
    return DLLM_OK;
}

DLLM_EXPORT int dllm_spherical_kmeans(const float *X, float *C, int32_t *assign, float *xnorm, int B, int N,
                                      int D, int K, int iters, void *stream) {
    CHECK_ARG(X && C && assign && xnorm, "null pointer");
    CHECK_ARG(B > 0 && N > 0 && D > 0 && K > 0 && iters >= 0, "sizes must be positive, iters >= 0");
    CHECK_ARG(B <= 65535, "B must be <= 65535");
    if (D > 8192 || D % 4 || K > 256)
        return fail(DLLM_ERR_UNSUPPORTED, "D must be a multiple of 4 up to 8192 and K <= 256 (D=%d K=%d)", D, K);
    CHECK_ARG(aligned16(X) && aligned16(C), "X and C must be 16-byte aligned");
    cudaStream_t st = as_stream(stream);
    Launch t(DLLM_KERNEL_CLUSTER, st, 2 * iters + 2);
    CHECK_CUDA(spherical_kmeans(X, C, assign, xnorm, B, N, D, K, iters, st), "k-means launch");
    return DLLM_OK;
}

DLLM_EXPORT int dllm_cluster_residual(const float *X, const float *C, const int32_t *assign, const float *xnorm,
                                      float *R, int B, int N, int D, int K, void *stream) {
    CHECK_ARG(X && C && assign && xnorm && R, "null pointer");
    CHECK_ARG(B > 0 && N > 0 && D > 0 && K > 0, "sizes must be positive");
    cudaStream_t st = as_stream(stream);
    Launch t(DLLM_KERNEL_CLUSTER, st);
    CHECK_CUDA(cluster_residual(X, C, assign, xnorm, R, B, N, D, K, st), "residual launch");
    return DLLM_OK;
}

DLLM_EXPORT int dllm_nvfp4_quantize(const float *R, float g, uint8_t *codes, uint8_t *scales, long rows, int D,
                                    void *stream) {
    CHECK_ARG(R && codes && scales, "null pointer");
    CHECK_ARG(rows > 0 && D > 0, "sizes must be positive");
    CHECK_ARG(g > 0.f && isfinite(g), "the tensor scale g must be positive and finite");
    CHECK_ARG(aligned16(R) && aligned8(codes), "R must be 16-byte and codes 8-byte aligned");
    if (D % 16) return fail(DLLM_ERR_UNSUPPORTED, "D must be a multiple of 16 (got %d)", D);
    cudaStream_t st = as_stream(stream);
    Launch t(DLLM_KERNEL_CLUSTER, st);
    CHECK_CUDA(nvfp4_quantize(R, g, codes, scales, rows, D, st), "NVFP4 launch");
    return DLLM_OK;
}

DLLM_EXPORT int dllm_nvfp4_dequantize(const uint8_t *codes, const uint8_t *scales, float g, float *out, long rows,
                                      int D, void *stream) {
    CHECK_ARG(codes && scales && out, "null pointer");
    CHECK_ARG(rows > 0 && D > 0, "sizes must be positive");
    CHECK_ARG(g > 0.f && isfinite(g), "the tensor scale g must be positive and finite");
    CHECK_ARG(aligned8(codes) && aligned16(out), "codes must be 8-byte and out 16-byte aligned");
    if (D % 16) return fail(DLLM_ERR_UNSUPPORTED, "D must be a multiple of 16 (got %d)", D);
    cudaStream_t st = as_stream(stream);
    Launch t(DLLM_KERNEL_CLUSTER, st);
    CHECK_CUDA(nvfp4_dequantize(codes, scales, g, out, rows, D, st), "NVFP4 dequantize launch");
    return DLLM_OK;
}

DLLM_EXPORT int dllm_cluster_select(const float *C_now, const float *C_prev, const int32_t *assign, int kc,
                                    int32_t *idx, int32_t *count, int B, int N, int D, int K, void *stream) {
    CHECK_ARG(C_now && C_prev && assign && idx && count, "null pointer");
    CHECK_ARG(B > 0 && N > 0 && D > 0 && K > 0 && kc >= 0, "sizes must be positive, kc >= 0");
    if (K > 256) return fail(DLLM_ERR_UNSUPPORTED, "K must be <= 256 (got %d)", K);
    cudaStream_t st = as_stream(stream);
    Launch t(DLLM_KERNEL_CLUSTER, st);
    CHECK_CUDA(cluster_select(C_now, C_prev, assign, kc, idx, count, B, N, D, K, st), "cluster select launch");
    return DLLM_OK;
}

// ------------------------------------------------------------------ selection
DLLM_EXPORT int dllm_select_topk(const float *drift, const int32_t *forced, int F, int k,
                                 float min_drift, int32_t *idx, int32_t *count, int B, int N,
                                 void *stream) {
    CHECK_ARG(drift && idx && count, "null pointer");
    CHECK_ARG(B > 0 && N > 0, "B and N must be positive");
    CHECK_ARG(N <= 16384, "N must be <= 16384 (got %d)", N);
    CHECK_ARG(k >= 0, "k must be >= 0");
    if (!forced) F = 0;
    CHECK_ARG(F >= 0, "F must be >= 0");
    Launch t(DLLM_KERNEL_SELECT, as_stream(stream));
    CHECK_CUDA(select_topk(drift, forced, F, k, min_drift, idx, count, B, N, as_stream(stream)),
               "select launch");
    return DLLM_OK;
}

DLLM_EXPORT double dllm_layer_rho(int l, double base, double peak, double centre, double sigma_left,
                                  double sigma_right) {
    const double s = (double)l < centre ? sigma_left : sigma_right;
    const double z = ((double)l - centre) / s;
    return base + (peak - base) * std::exp(-0.5 * z * z);
}

DLLM_EXPORT int dllm_layer_budget(double rho, int N) {
    if (!(rho > 0.0) || N <= 0) return 0;
    double k = std::ceil(rho * (double)N);
    if (k < 1.0) k = 1.0;
    if (k > (double)N) k = (double)N;
    return (int)k;
}

// ------------------------------------------------------------------ weights
DLLM_EXPORT size_t dllm_packed_layer_bytes(int d, int n_q, int n_kv, int hd, int F, int dtype) {
    if (d <= 0 || n_q <= 0 || n_kv <= 0 || hd <= 0 || F <= 0) return 0;
    return pack_layout(d, n_q, n_kv, hd, F, dtype).total;
}

DLLM_EXPORT int dllm_pack_layer(const void *w_q, const void *w_k, const void *w_v, const void *w_o,
                                const void *w_g, const void *w_u, const void *w_d,
                                const void *gamma1, const void *gamma2, int d, int n_q, int n_kv,
                                int hd, int F, float eps, float rope_theta, int use_rope, int dtype,
                                void *dst, size_t dst_bytes, dllm_layer *out, void *stream) {
    CHECK_ARG(w_q && w_k && w_v && w_o && w_g && w_u && w_d && gamma1 && gamma2 && dst && out,
              "null pointer");
    CHECK_ARG(dtype == DLLM_BF16 || dtype == DLLM_F32, "dtype must be DLLM_BF16 or DLLM_F32");
    CHECK_ARG(d > 0 && n_q > 0 && n_kv > 0 && F > 0, "sizes must be positive");
    if (hd != 64 && hd != 128) return fail(DLLM_ERR_UNSUPPORTED, "hd must be 64 or 128 (got %d)", hd);
    CHECK_ARG(n_q % n_kv == 0, "n_q must be a multiple of n_kv");
    CHECK_ARG(rope_theta > 0.f, "rope_theta must be positive");
    CHECK_ARG((reinterpret_cast<uintptr_t>(dst) & 255u) == 0, "dst must be 256-byte aligned");
    const PackLayout L = pack_layout(d, n_q, n_kv, hd, F, dtype);
    if (dst_bytes < L.total)
        return fail(DLLM_ERR_WORKSPACE, "dst holds %zu bytes, %zu needed", dst_bytes, L.total);
    cudaStream_t st = as_stream(stream);
    uint8_t *base = static_cast<uint8_t *>(dst);
    const size_t el = el_size(dtype);
    const size_t dq = (size_t)n_q * hd, dkv = (size_t)n_kv * hd;
    uint8_t *qkv = base + L.qkv;
    if (dtype == DLLM_BF16) {
        CHECK_CUDA(pack_rows_rope(static_cast<const bf16 *>(w_q), reinterpret_cast<bf16 *>(qkv), (int)dq, d, hd, st), "pack q");
        CHECK_CUDA(pack_rows_rope(static_cast<const bf16 *>(w_k), reinterpret_cast<bf16 *>(qkv + dq * d * el), (int)dkv, d, hd, st), "pack k");
        CHECK_CUDA(pack_rows_rope(static_cast<const bf16 *>(w_v), reinterpret_cast<bf16 *>(qkv + (dq + dkv) * d * el), (int)dkv, d, hd, st), "pack v");
        CHECK_CUDA(pack_rows_interleave(static_cast<const bf16 *>(w_g), static_cast<const bf16 *>(w_u), reinterpret_cast<bf16 *>(base + L.gu), F, d, st), "pack gate/up");
    } else {
        CHECK_CUDA(pack_rows_rope(static_cast<const float *>(w_q), reinterpret_cast<float *>(qkv), (int)dq, d, hd, st), "pack q");
        CHECK_CUDA(pack_rows_rope(static_cast<const float *>(w_k), reinterpret_cast<float *>(qkv + dq * d * el), (int)dkv, d, hd, st), "pack k");
        CHECK_CUDA(pack_rows_rope(static_cast<const float *>(w_v), reinterpret_cast<float *>(qkv + (dq + dkv) * d * el), (int)dkv, d, hd, st), "pack v");
        CHECK_CUDA(pack_rows_interleave(static_cast<const float *>(w_g), static_cast<const float *>(w_u), reinterpret_cast<float *>(base + L.gu), F, d, st), "pack gate/up");
    }
    CHECK_CUDA(cudaMemcpyAsync(base + L.o, w_o, (size_t)d * dq * el, cudaMemcpyDeviceToDevice, st), "copy w_o");
    CHECK_CUDA(cudaMemcpyAsync(base + L.down, w_d, (size_t)d * F * el, cudaMemcpyDeviceToDevice, st), "copy w_down");
    CHECK_CUDA(cudaMemcpyAsync(base + L.g1, gamma1, (size_t)d * el, cudaMemcpyDeviceToDevice, st), "copy gamma1");
    CHECK_CUDA(cudaMemcpyAsync(base + L.g2, gamma2, (size_t)d * el, cudaMemcpyDeviceToDevice, st), "copy gamma2");
    CHECK_CUDA(rope_inv_freq(reinterpret_cast<float *>(base + L.freq), hd, rope_theta, st), "rotary table");
    out->w_qkv = base + L.qkv;
    out->w_o = base + L.o;
    out->w_gu = base + L.gu;
    out->w_down = base + L.down;
    out->gamma1 = base + L.g1;
    out->gamma2 = base + L.g2;
    out->rope_inv_freq = reinterpret_cast<const float *>(base + L.freq);
    out->d = d;
    out->n_q = n_q;
    out->n_kv = n_kv;
    out->hd = hd;
    out->F = F;
    out->eps = eps;
    out->rope_theta = rope_theta;
    out->use_rope = use_rope ? 1 : 0;
    out->dtype = dtype;
    return DLLM_OK;
}

// ------------------------------------------------------------------ sparse refresh
DLLM_EXPORT size_t dllm_refresh_workspace_bytes(const dllm_layer *W, int B, int N, int k_max) {
    if (!W || B <= 0 || N <= 0 || k_max <= 0) return 0;
    return refresh_ws(W, B, N, k_max).total;
}

namespace {

// The per-layer step's selection arguments, when the selection is fused with the gather
// (and, with dp.parts set, preceded by the drift computed from the projection's partials).
struct FusedSelect {
    float *drift;
    const int32_t *forced;
    int F, k;
    float min_drift;
    int32_t *idx, *count;
    DriftParts dp;
};

template <class T>
int refresh_impl(const dllm_layer *W, const T *H_in, SelRows sel, int B, T *K_cache, T *V_cache,
                 T *H_out, float *proxy_cache, float *proxy_cur, int r, uint8_t *ws,
                 cudaStream_t st, const FusedSelect *fs = nullptr) {
    const RefreshWs L = refresh_ws(W, B, sel.N, sel.k_max);
    const int M = B * sel.k_max;
    const int d = W->d, dq = W->n_q * W->hd, dkv = W->n_kv * W->hd, F = W->F;
    T *Xn = reinterpret_cast<T *>(ws + L.xn);
    T *Qc = reinterpret_cast<T *>(ws + L.q);
    T *Ac = reinterpret_cast<T *>(ws + L.a);
    float *h1 = reinterpret_cast<float *>(ws + L.h1);
    float2 *rope_cs = W->use_rope ? reinterpret_cast<float2 *>(ws + L.rope) : nullptr;
    T *Xn2 = reinterpret_cast<T *>(ws + L.xn2);
    T *U = reinterpret_cast<T *>(ws + L.u);
    unsigned *status = status_ptr();
    const T *wqkv = static_cast<const T *>(W->w_qkv);
    const T *wo = static_cast<const T *>(W->w_o);
    const T *wgu = static_cast<const T *>(W->w_gu);
    const T *wdn = static_cast<const T *>(W->w_down);
    const T *g1 = static_cast<const T *>(W->gamma1);
    const T *g2 = static_cast<const T *>(W->gamma2);

    // a2 + a3 fused (the layer step): selection, then gather + RMSNorm, proxy cache update
    if (fs) {
        Launch t(DLLM_KERNEL_SELECT, st);
        CHECK_CUDA(select_gather<T>(fs->drift, fs->forced, fs->F, fs->k, fs->min_drift, fs->idx, fs->count, B, sel.N,
                                    sel.k_max, H_in, d, g1, W->eps, Xn, proxy_cache, proxy_cur, r, W->rope_inv_freq,
                                    W->hd / 2, rope_cs, fs->dp, status, st),
                   "select + gather launch");
    } else {   // a3: gather + RMSNorm, proxy cache update
        Launch t(DLLM_KERNEL_GATHER, st);
        CHECK_CUDA(gather_rmsnorm<T>(H_in, sel, B, d, g1, W->eps, Xn, proxy_cache, proxy_cur, r,
                                     W->rope_inv_freq, W->hd / 2, rope_cs, status, st),
                   "gather launch");
    }
    // a4: QKV projection, rotary embedding, K/V scattered into the cache
    EpiQKV<T> eq{sel, Qc, K_cache, V_cache, rope_cs, W->n_q, W->n_kv, W->hd, W->use_rope};
    // a6: O projection + residual;  a7: FFN gate/up + SwiGLU;  a8: down + residual, scattered
    EpiResidual<T> er{sel, h1, H_in, d};
    EpiSwiGLU<T> es{SelRows{}, U, F};
    EpiDownScatter<T> ed{sel, H_out, h1, d};
    if constexpr (sizeof(T) == 2) {
        { Launch t(DLLM_KERNEL_QKV, st); CHECK_CUDA(gemm_tc(wqkv, dq + 2 * dkv, d, Xn, M, eq, 0, true, status, st), "qkv gemm"); }
        {
            const int na = 1;
            Launch t(DLLM_KERNEL_ATTENTION, st, na);
            CHECK_CUDA(attention_tc(reinterpret_cast<const bf16 *>(Qc), reinterpret_cast<const bf16 *>(K_cache),
                                    reinterpret_cast<const bf16 *>(V_cache), reinterpret_cast<bf16 *>(Ac), sel, B,
                                    W->n_q, W->n_kv, W->hd, status, st),
                       "attention");
        }
        if (M <= kFoldNormRows) {
            // a6 + a7, few rows: the second RMSNorm folded into the O epilogue (bf16 h1 * gamma2
            // and the rows' partial squares) and into the gate/up epilogue (1 / rms): one
            // launch fewer where every launch's fixed cost counts
            float *ss = reinterpret_cast<float *>(ws + L.ss);
            EpiResidualNorm<T> ern{sel, h1, Xn2, ss, H_in, g2, d, M};
            EpiSwiGLUNorm<T> esn{SelRows{}, U, ss, F, d, M, W->eps};
            { Launch t(DLLM_KERNEL_OPROJ, st); CHECK_CUDA(gemm_tc(wo, d, dq, Ac, M, ern, 0, true, status, st), "o gemm"); }
            { Launch t(DLLM_KERNEL_GATEUP, st); CHECK_CUDA(gemm_tc(wgu, 2 * F, d, Xn2, M, esn, 0, true, status, st), "gate/up gemm"); }
        } else {
            // many rows: the heavier epilogues cost more than the norm kernel they replace
            { Launch t(DLLM_KERNEL_OPROJ, st); CHECK_CUDA(gemm_tc(wo, d, dq, Ac, M, er, 0, true, status, st), "o gemm"); }
            { Launch t(DLLM_KERNEL_RMSNORM2, st); CHECK_CUDA(rmsnorm_rows<T>(h1, M, d, g2, W->eps, Xn2, st), "rmsnorm2"); }
            { Launch t(DLLM_KERNEL_GATEUP, st); CHECK_CUDA(gemm_tc(wgu, 2 * F, d, Xn2, M, es, 0, true, status, st), "gate/up gemm"); }
        }
        { Launch t(DLLM_KERNEL_DOWN, st); CHECK_CUDA(gemm_tc(wdn, d, F, U, M, ed, 0, true, status, st), "down gemm"); }
    } else {
        { Launch t(DLLM_KERNEL_QKV, st); CHECK_CUDA(gemm_simt(wqkv, dq + 2 * dkv, d, Xn, M, eq, st), "qkv gemm"); }
        { Launch t(DLLM_KERNEL_ATTENTION, st); CHECK_CUDA(attention_simt<T>(Qc, K_cache, V_cache, Ac, sel, B, W->n_q, W->n_kv, W->hd, st), "attention"); }
        { Launch t(DLLM_KERNEL_OPROJ, st); CHECK_CUDA(gemm_simt(wo, d, dq, Ac, M, er, st), "o gemm"); }
        { Launch t(DLLM_KERNEL_RMSNORM2, st); CHECK_CUDA(rmsnorm_rows<T>(h1, M, d, g2, W->eps, Xn2, st), "rmsnorm2"); }
        { Launch t(DLLM_KERNEL_GATEUP, st); CHECK_CUDA(gemm_simt(wgu, 2 * F, d, Xn2, M, es, st), "gate/up gemm"); }
        { Launch t(DLLM_KERNEL_DOWN, st); CHECK_CUDA(gemm_simt(wdn, d, F, U, M, ed, st), "down gemm"); }
    }
    return DLLM_OK;
}

}  // namespace

DLLM_EXPORT int dllm_sparse_layer_refresh(const dllm_layer *W, const void *H_in,
                                          const int32_t *idx, const int32_t *count, int k_max,
                                          void *K_cache, void *V_cache, void *H_out_cache,
                                          float *proxy_cache, const float *proxy_cur, int r, int B,
                                          int N, void *ws, size_t ws_bytes, void *stream) {
    int rc = check_layer(W);
    if (rc != DLLM_OK) return rc;
    CHECK_ARG(H_in && idx && count && K_cache && V_cache && H_out_cache, "null pointer");
    CHECK_ARG(B > 0 && N > 0, "B and N must be positive");
    CHECK_ARG(k_max >= 0 && k_max <= N, "k_max must be in [0, N] (got %d, N=%d)", k_max, N);
    CHECK_ARG(H_out_cache != H_in, "H_out_cache must not alias H_in");
    CHECK_ARG(aligned16(H_in) && aligned16(K_cache) && aligned16(V_cache) && aligned16(H_out_cache),
              "arrays must be 16-byte aligned");
    CHECK_ARG(W->rope_inv_freq || !W->use_rope, "rope table missing (use dllm_pack_layer)");
    if ((proxy_cache != nullptr) != (proxy_cur != nullptr))
        return fail(DLLM_ERR_INVALID_ARG, "proxy_cache and proxy_cur must both be set or both NULL");
    if (proxy_cache) CHECK_ARG(r > 0, "r must be positive when proxies are given");
    if (k_max == 0) return DLLM_OK;
    const size_t need = refresh_ws(W, B, N, k_max).total;
    if (!ws || ws_bytes < need)
        return fail(DLLM_ERR_WORKSPACE, "workspace holds %zu bytes, %zu needed", ws_bytes, need);
    uint8_t *w8 = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(ws) + 255) & ~uintptr_t(255));
    SelRows sel{idx, count, k_max, N};
    cudaStream_t st = as_stream(stream);
    // (without a fused selection the refresh only reads proxy_cur)
    float *cur = const_cast<float *>(proxy_cur);
    if (W->dtype == DLLM_BF16)
        return refresh_impl<bf16>(W, static_cast<const bf16 *>(H_in), sel, B, static_cast<bf16 *>(K_cache),
                                  static_cast<bf16 *>(V_cache), static_cast<bf16 *>(H_out_cache),
                                  proxy_cache, cur, r, w8, st);
    return refresh_impl<float>(W, static_cast<const float *>(H_in), sel, B, static_cast<float *>(K_cache),
                               static_cast<float *>(V_cache), static_cast<float *>(H_out_cache),
                               proxy_cache, cur, r, w8, st);
}

// ------------------------------------------------------------------ one layer step
DLLM_EXPORT size_t dllm_layer_step_workspace_bytes(const dllm_layer *W, int B, int N, int r, int F, int k) {
    if (!W || B <= 0 || N <= 0 || r <= 0 || F < 0 || k < 0) return 0;
    const long long km = (long long)k + F < N ? (long long)k + F : N;
    const int k_max = km > 0 ? (int)km : 1;
    // refresh scratch, the proxy projection's partials, the selection's arrival counters
    return refresh_ws(W, B, N, k_max).total + dllm_proxy_workspace_bytes(B, N, W->d, r, W->dtype) +
           (size_t)B * sizeof(unsigned) + 256 + 256;
}

DLLM_EXPORT int dllm_layer_step(const dllm_layer *W, const void *Pt, const void *H_in, float *proxy_cache,
                                float *proxy_cur, float *drift, const int32_t *forced, int F, int k, float min_drift,
                                int32_t *idx, int32_t *count, void *K_cache, void *V_cache, void *H_out_cache,
                                int B, int N, int r, void *ws, size_t ws_bytes, void *stream) {
    int rc = check_layer(W);
    if (rc != DLLM_OK) return rc;
    CHECK_ARG(Pt && H_in && proxy_cache && proxy_cur && drift && idx && count && K_cache && V_cache && H_out_cache,
              "null pointer");
    CHECK_ARG(B > 0 && N > 0 && r > 0, "sizes must be positive (B=%d N=%d r=%d)", B, N, r);
    CHECK_ARG(N <= 16384, "N must be <= 16384 (got %d)", N);
    CHECK_ARG(k >= 0, "k must be >= 0");
    if (!forced) F = 0;
    CHECK_ARG(F >= 0, "F must be >= 0");
    CHECK_ARG((long long)B * N <= INT_MAX, "B*N must fit in an int");
    CHECK_ARG(H_out_cache != H_in, "H_out_cache must not alias H_in");
    CHECK_ARG(aligned16(H_in) && aligned16(K_cache) && aligned16(V_cache) && aligned16(H_out_cache) &&
                  aligned16(Pt) && aligned16(proxy_cache) && aligned16(proxy_cur),
              "arrays must be 16-byte aligned");
    CHECK_ARG(W->rope_inv_freq || !W->use_rope, "rope table missing (use dllm_pack_layer)");
    const int k_max = (int)((long long)k + F < N ? (long long)k + F : N);
    const size_t need = dllm_layer_step_workspace_bytes(W, B, N, r, F, k);
    if (!ws || ws_bytes < need)
        return fail(DLLM_ERR_WORKSPACE, "workspace holds %zu bytes, %zu needed", ws_bytes, need);
    cudaStream_t st = as_stream(stream);
    // a1: proxy + drift (its K-slice partials, where it needs them, after the refresh scratch)
    const size_t rws = k_max > 0 ? refresh_ws(W, B, N, k_max).total : 0;
    uint8_t *w8 = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(ws) + 255) & ~uintptr_t(255));
    const int nparts = proxy_slices(B, N, W->d, r, W->dtype);
    // a selection fused with the gather that also computes the drift (no cosine kernel):
    // from the bf16 projection's K-slice partials, or from the fp32 projection's proxies;
    // the projection clears the selection's per-sequence arrival counters, placed after
    // the partials
    const DriftParts no_parts{nullptr, 0, nullptr};
    DriftParts dp = no_parts;
    const bool front_fused = (W->dtype == DLLM_F32 || nparts > 1) && r <= 128 && k_max > 0 &&
                             N <= select_gather_max_n() && select_gather_fused_ok(B, N, k_max, W->dtype);
    if (front_fused) {
        const size_t pbytes = dllm_proxy_workspace_bytes(B, N, W->d, r, W->dtype);
        unsigned *arrive = reinterpret_cast<unsigned *>(w8 + rws + pbytes);
        Launch t(DLLM_KERNEL_PROXY_GEMM, st);
        if (W->dtype == DLLM_BF16) {
            float *parts = reinterpret_cast<float *>(
                (reinterpret_cast<uintptr_t>(w8 + rws) + 255) & ~uintptr_t(255));
            dp = DriftParts{parts, nparts, arrive};
            CHECK_CUDA(gemm_tc_slices(static_cast<const bf16 *>(Pt), r, W->d, static_cast<const bf16 *>(H_in),
                                      B * N, parts, true, status_ptr(), st, arrive, B),
                       "proxy projection launch");
        } else {   // one fp32 product straight into proxy_cur
            dp = DriftParts{proxy_cur, 1, arrive};
            EpiStoreF32 epi{SelRows{}, proxy_cur, r, r};
            CHECK_CUDA(gemm_simt(static_cast<const float *>(Pt), r, W->d, static_cast<const float *>(H_in), B * N,
                                 epi, st, arrive, B),
                       "proxy projection launch");
        }
    } else {
        rc = dllm_proxy_score(H_in, Pt, proxy_cache, proxy_cur, drift, B, N, W->d, r, W->dtype, w8 + rws,
                              ws_bytes - rws - 256, stream);
        if (rc != DLLM_OK) return rc;
    }
    if (k_max == 0) {   // nothing can be selected: empty selection
        return dllm_select_topk(drift, forced, F, k, min_drift, idx, count, B, N, stream);
    }
    SelRows sel{idx, count, k_max, N};
    if (N > select_gather_max_n()) {   // long sequences: the selection kernel, then the plain refresh
        rc = dllm_select_topk(drift, forced, F, k, min_drift, idx, count, B, N, stream);
        if (rc != DLLM_OK) return rc;
        if (W->dtype == DLLM_BF16)
            return refresh_impl<bf16>(W, static_cast<const bf16 *>(H_in), sel, B, static_cast<bf16 *>(K_cache),
                                      static_cast<bf16 *>(V_cache), static_cast<bf16 *>(H_out_cache), proxy_cache,
                                      proxy_cur, r, w8, st);
        return refresh_impl<float>(W, static_cast<const float *>(H_in), sel, B, static_cast<float *>(K_cache),
                                   static_cast<float *>(V_cache), static_cast<float *>(H_out_cache), proxy_cache,
                                   proxy_cur, r, w8, st);
    }
    const FusedSelect fs{drift, forced, F, k, min_drift, idx, count, dp};
    if (W->dtype == DLLM_BF16)
        return refresh_impl<bf16>(W, static_cast<const bf16 *>(H_in), sel, B, static_cast<bf16 *>(K_cache),
                                  static_cast<bf16 *>(V_cache), static_cast<bf16 *>(H_out_cache), proxy_cache,
                                  proxy_cur, r, w8, st, &fs);
    return refresh_impl<float>(W, static_cast<const float *>(H_in), sel, B, static_cast<float *>(K_cache),
                               static_cast<float *>(V_cache), static_cast<float *>(H_out_cache), proxy_cache,
                               proxy_cur, r, w8, st, &fs);
}

// ------------------------------------------------------------------ attention alone
DLLM_EXPORT size_t dllm_attention_workspace_bytes(int B, int N, int k_max, int n_q, int hd, int dtype) {
    (void)B; (void)N; (void)k_max; (void)n_q; (void)hd; (void)dtype;
    return 0;   // the key-range split is merged on chip
}

DLLM_EXPORT int dllm_attention(const void *Q, const void *K_cache, const void *V_cache, void *A,
                               const int32_t *idx, const int32_t *count, int k_max, int B, int N,
                               int n_q, int n_kv, int hd, int dtype, void *ws, size_t ws_bytes,
                               void *stream) {
    CHECK_ARG(Q && K_cache && V_cache && A && idx && count, "null pointer");
    CHECK_ARG(B > 0 && N > 0 && n_q > 0 && n_kv > 0, "sizes must be positive");
    CHECK_ARG(k_max > 0 && k_max <= N, "k_max must be in [1, N]");
    CHECK_ARG(n_q % n_kv == 0, "n_q must be a multiple of n_kv");
    CHECK_ARG(dtype == DLLM_BF16 || dtype == DLLM_F32, "dtype must be DLLM_BF16 or DLLM_F32");
    if (hd != 64 && hd != 128) return fail(DLLM_ERR_UNSUPPORTED, "hd must be 64 or 128 (got %d)", hd);
    CHECK_ARG(aligned16(Q) && aligned16(K_cache) && aligned16(V_cache) && aligned16(A),
              "arrays must be 16-byte aligned");
    const size_t need = dllm_attention_workspace_bytes(B, N, k_max, n_q, hd, dtype);
    if (need > 0 && (!ws || ws_bytes < need))
        return fail(DLLM_ERR_WORKSPACE, "workspace holds %zu bytes, %zu needed", ws_bytes, need);
    SelRows sel{idx, count, k_max, N};
    cudaStream_t st = as_stream(stream);
    Launch t(DLLM_KERNEL_ATTENTION, st);
    cudaError_t e;
    if (dtype == DLLM_BF16) {
        e = attention_tc(static_cast<const bf16 *>(Q), static_cast<const bf16 *>(K_cache),
                         static_cast<const bf16 *>(V_cache), static_cast<bf16 *>(A), sel, B, n_q, n_kv, hd,
                         status_ptr(), st);
    } else {
        e = attention_simt(static_cast<const float *>(Q), static_cast<const float *>(K_cache),
                           static_cast<const float *>(V_cache), static_cast<float *>(A), sel, B, n_q, n_kv,
                           hd, st);
    }
    CHECK_CUDA(e, "attention launch");
    return DLLM_OK;
}

// ------------------------------------------------------------------ embedding, final norm
DLLM_EXPORT int dllm_embed(const void *E, const int32_t *tokens, const int32_t *rows, int R, void *H,
                           int B, int N, int d, int V, int dtype, void *stream) {
    CHECK_ARG(E && tokens && H, "null pointer");
    CHECK_ARG(B > 0 && N > 0 && d > 0 && V > 0, "sizes must be positive");
    CHECK_ARG(!rows || R >= 0, "R must be >= 0");
    CHECK_ARG(dtype == DLLM_BF16 || dtype == DLLM_F32, "dtype must be DLLM_BF16 or DLLM_F32");
    cudaStream_t st = as_stream(stream);
    Launch t(DLLM_KERNEL_GATHER, st);
    cudaError_t e = dtype == DLLM_BF16
                        ? embed_rows(static_cast<const bf16 *>(E), tokens, rows, R, static_cast<bf16 *>(H), B, N, d, V, st)
                        : embed_rows(static_cast<const float *>(E), tokens, rows, R, static_cast<float *>(H), B, N, d, V, st);
    CHECK_CUDA(e, "embed launch");
    return DLLM_OK;
}

DLLM_EXPORT int dllm_rows_rmsnorm(const void *H, const int32_t *rows, int R, const void *gamma,
                                  float eps, void *out, int B, int N, int d, int dtype, void *stream) {
    CHECK_ARG(H && rows && gamma && out, "null pointer");
    CHECK_ARG(B > 0 && N > 0 && d > 0 && R >= 0, "bad sizes");
    CHECK_ARG(dtype == DLLM_BF16 || dtype == DLLM_F32, "dtype must be DLLM_BF16 or DLLM_F32");
    cudaStream_t st = as_stream(stream);
    Launch t(DLLM_KERNEL_RMSNORM2, st);
    cudaError_t e = dtype == DLLM_BF16
                        ? rows_rmsnorm(static_cast<const bf16 *>(H), rows, R, static_cast<const bf16 *>(gamma), eps,
                                       static_cast<bf16 *>(out), B, N, d, st)
                        : rows_rmsnorm(static_cast<const float *>(H), rows, R, static_cast<const float *>(gamma), eps,
                                       static_cast<float *>(out), B, N, d, st);
    CHECK_CUDA(e, "rows rmsnorm launch");
    return DLLM_OK;
}

DLLM_EXPORT int dllm_gather_rows(const void *src, const int32_t *idx, const int32_t *count, int k_max, void *dst,
                                 int B, int N, int row_bytes, void *stream) {
    CHECK_ARG(src && idx && count && dst, "null pointer");
    CHECK_ARG(B > 0 && N > 0 && row_bytes > 0, "sizes must be positive");
    CHECK_ARG(k_max > 0 && k_max <= N, "k_max must be in [1, N] (got %d, N=%d)", k_max, N);
    CHECK_ARG((long long)B * k_max <= INT_MAX, "B*k_max must fit in an int");
    CHECK_ARG(row_bytes % 16 == 0, "row_bytes must be a multiple of 16 (got %d)", row_bytes);
    CHECK_ARG(aligned16(src) && aligned16(dst), "src and dst must be 16-byte aligned");
    cudaStream_t st = as_stream(stream);
    GatherSet gs{};
    gs.src[0] = src;
    gs.dst[0] = dst;
    gs.vecs[0] = row_bytes / 16;
    Launch t(DLLM_KERNEL_GATHER, st);
    CHECK_CUDA(gather_rows(gs, 1, SelRows{idx, count, k_max, N}, B, st), "gather rows launch");
    return DLLM_OK;
}

DLLM_EXPORT int dllm_gather_rows_n(int n, const void *const *srcs, void *const *dsts, const int *row_bytes,
                                   const int32_t *idx, const int32_t *count, int k_max, int B, int N,
                                   void *stream) {
    CHECK_ARG(srcs && dsts && row_bytes && idx && count, "null pointer");
    CHECK_ARG(n >= 1 && n <= kGatherMax, "n must be in [1, %d] (got %d)", kGatherMax, n);
    CHECK_ARG(B > 0 && N > 0, "sizes must be positive");
    CHECK_ARG(k_max > 0 && k_max <= N, "k_max must be in [1, N] (got %d, N=%d)", k_max, N);
    CHECK_ARG((long long)B * k_max <= INT_MAX, "B*k_max must fit in an int");
    GatherSet gs{};
    for (int t = 0; t < n; ++t) {
        CHECK_ARG(srcs[t] && dsts[t], "null pointer (cache %d)", t);
        CHECK_ARG(row_bytes[t] > 0 && row_bytes[t] % 16 == 0,
                  "row_bytes[%d] must be a positive multiple of 16 (got %d)", t, row_bytes[t]);
        CHECK_ARG(aligned16(srcs[t]) && aligned16(dsts[t]), "cache %d: src and dst must be 16-byte aligned", t);
        gs.src[t] = srcs[t];
        gs.dst[t] = dsts[t];
        gs.vecs[t] = row_bytes[t] / 16;
    }
    cudaStream_t st = as_stream(stream);
    Launch t(DLLM_KERNEL_GATHER, st);
    CHECK_CUDA(gather_rows(gs, n, SelRows{idx, count, k_max, N}, B, st), "gather rows launch");
    return DLLM_OK;
}

// ------------------------------------------------------------------ plain GEMM
DLLM_EXPORT int dllm_gemm_bf16(const void *X, const void *W, float *out, int M, int N_out, int K,
                               int splits, void *stream) {
    CHECK_ARG(X && W && out, "null pointer");
    CHECK_ARG(M > 0 && N_out > 0 && K > 0, "sizes must be positive");
    CHECK_ARG(splits >= 0 && splits <= 8, "splits must be in [0, 8]");
    CHECK_ARG(aligned16(X) && aligned16(W) && aligned16(out), "arrays must be 16-byte aligned");
    if (K % 64 || N_out % 32) return fail(DLLM_ERR_UNSUPPORTED, "needs K %% 64 == 0 and N_out %% 32 == 0");
    cudaStream_t st = as_stream(stream);
    Launch t(DLLM_KERNEL_GEMM, st);
    EpiStoreF32 epi{SelRows{}, out, N_out, N_out};
    CHECK_CUDA(gemm_tc(static_cast<const bf16 *>(W), N_out, K, static_cast<const bf16 *>(X), M, epi,
                       splits, false, status_ptr(), st),
               "gemm launch");
    return DLLM_OK;
}

DLLM_EXPORT int dllm_gemm_plan(int M, int N_out, int K, int splits, int sms, int slices, int32_t *info) {
    CHECK_ARG(info, "null pointer");
    CHECK_ARG(M > 0 && N_out > 0 && K > 0, "sizes must be positive");
    CHECK_ARG(sms >= 1 && sms <= 1024, "sms must be in [1, 1024] (got %d)", sms);
    CHECK_ARG(splits >= 0 && splits <= 8, "splits must be in [0, 8]");
    if (K % 64 || N_out % 32) return fail(DLLM_ERR_UNSUPPORTED, "needs K %% 64 == 0 and N_out %% 32 == 0");
    int v[8];
    CHECK_ARG(slices >= 0 && slices <= 2, "slices must be 0, 1 or 2 (got %d)", slices);
    if (gemm_tc_plan_info(M, N_out, K, splits, sms, slices, v) != 0)
        return fail(DLLM_ERR_INVALID_ARG, "shape rejected by the planner");
    for (int i = 0; i < 8; ++i) info[i] = v[i];
    return DLLM_OK;
}

// ------------------------------------------------------------------ vocabulary
DLLM_EXPORT size_t dllm_commit_workspace_bytes(int B, int M, int V) {
    if (B <= 0 || M < 0 || V <= 0 || (long long)B * M > INT_MAX) return 0;
    return commit_ws_bytes(B, M, V) + 256;
}

DLLM_EXPORT int dllm_commit_entropy(const float *logits, const uint8_t *valid, int B, int M, int V,
                                    float conf_thresh, float tau, int32_t *token, float *conf,
                                    float *entropy, float *max_entropy, int32_t *full_next,
                                    void *ws, size_t ws_bytes, void *stream) {
    CHECK_ARG(max_entropy && full_next, "null pointer");
    CHECK_ARG(B > 0 && M >= 0 && V > 0, "sizes must be positive");
    CHECK_ARG(M <= 1024, "M must be <= 1024 (got %d)", M);
    CHECK_ARG((long long)B * M <= INT_MAX, "B*M must fit in an int (B=%d M=%d)", B, M);
    if (M > 0) CHECK_ARG(logits && valid && token && conf && entropy, "null pointer");
    const size_t need = commit_ws_bytes(B, M, V) + 256;
    if (!ws || ws_bytes < need)
        return fail(DLLM_ERR_WORKSPACE, "workspace holds %zu bytes, %zu needed", ws_bytes, need);
    void *w = reinterpret_cast<void *>((reinterpret_cast<uintptr_t>(ws) + 255) & ~uintptr_t(255));
    Launch t(DLLM_KERNEL_VOCAB, as_stream(stream), 2);
    CHECK_CUDA(commit_entropy(logits, valid, B, M, V, conf_thresh, tau, token, conf, entropy,
                              max_entropy, full_next, w, as_stream(stream)),
               "commit launch");
    return DLLM_OK;
}

// ------------------------------------------------------------------ fused LM head + commit
namespace {
int vocab_tiles(int V) { return (V + 127) / 128; }
}  // namespace

DLLM_EXPORT size_t dllm_lmhead_workspace_bytes(int B, int M, int V) {
    if (B <= 0 || M <= 0 || V <= 0) return 0;
    return (size_t)B * M * vocab_tiles(V) * sizeof(VocabState) + 256;
}

DLLM_EXPORT int dllm_lmhead_commit(const void *X, const void *W_lm, const uint8_t *valid, int B, int M,
                                   int V, int d, float conf_thresh, float tau, int32_t *token, float *conf,
                                   float *entropy, float *max_entropy, int32_t *full_next, void *ws,
                                   size_t ws_bytes, void *stream) {
    CHECK_ARG(X && W_lm && valid && token && conf && entropy && max_entropy && full_next, "null pointer");
    CHECK_ARG(B > 0 && M > 0 && V > 0 && d > 0, "sizes must be positive");
    CHECK_ARG(M <= 1024, "M must be <= 1024 (got %d)", M);
    CHECK_ARG(aligned16(X) && aligned16(W_lm), "arrays must be 16-byte aligned");
    if (d % 64 || V % 32) return fail(DLLM_ERR_UNSUPPORTED, "needs d %% 64 == 0 and V %% 32 == 0");
    const size_t need = dllm_lmhead_workspace_bytes(B, M, V);
    if (!ws || ws_bytes < need)
        return fail(DLLM_ERR_WORKSPACE, "workspace holds %zu bytes, %zu needed", ws_bytes, need);
    VocabState *part = reinterpret_cast<VocabState *>((reinterpret_cast<uintptr_t>(ws) + 255) & ~uintptr_t(255));
    cudaStream_t st = as_stream(stream);
    const int tiles = vocab_tiles(V);
    {
        Launch t(DLLM_KERNEL_GEMM, st);
        EpiVocabStats epi{SelRows{}, part, tiles};
        CHECK_CUDA(gemm_tc(static_cast<const bf16 *>(W_lm), V, d, static_cast<const bf16 *>(X), B * M, epi, 1,
                           true, status_ptr(), st),
                   "lm head launch");
    }
    Launch t(DLLM_KERNEL_VOCAB, st);
    CHECK_CUDA(commit_from_states(part, tiles, valid, B, M, conf_thresh, tau, token, conf, entropy, max_entropy,
                                  full_next, st),
               "commit launch");
    return DLLM_OK;
}

// ------------------------------------------------------------------ measurement support
DLLM_EXPORT int dllm_timer_start(int kernel_id, int max_launches) {
    CHECK_ARG(kernel_id >= DLLM_KERNEL_PROXY_GEMM && kernel_id <= DLLM_KERNEL_CLUSTER, "unknown kernel id %d", kernel_id);
    CHECK_ARG(max_launches > 0 && max_launches <= 1 << 16, "max_launches must be in [1, 65536]");
    std::lock_guard<std::mutex> lock(g_timer.mu);
    CHECK_ARG(g_timer.armed == 0, "a timer is already armed");
    for (cudaEvent_t e : g_timer.ev) cudaEventDestroy(e);
    g_timer.ev.assign(2 * (size_t)max_launches, nullptr);
    for (auto &e : g_timer.ev) CHECK_CUDA(cudaEventCreate(&e), "cudaEventCreate");
    g_timer.cap = max_launches;
    g_timer.n = 0;
    g_timer.armed = kernel_id;
    return DLLM_OK;
}

DLLM_EXPORT int dllm_timer_stop(double *total_ms, int *launches) {
    std::lock_guard<std::mutex> lock(g_timer.mu);
    CHECK_ARG(g_timer.armed != 0, "no timer armed");
    g_timer.armed = 0;
    CHECK_CUDA(cudaDeviceSynchronize(), "cudaDeviceSynchronize");
    double tot = 0.0;
    for (int i = 0; i < g_timer.n; ++i) {
        float ms = 0.f;
        CHECK_CUDA(cudaEventElapsedTime(&ms, g_timer.ev[2 * i], g_timer.ev[2 * i + 1]), "cudaEventElapsedTime");
        tot += ms;
    }
    if (total_ms) *total_ms = tot;
    if (launches) *launches = g_timer.n;
    for (cudaEvent_t e : g_timer.ev) cudaEventDestroy(e);
    g_timer.ev.clear();
    g_timer.n = g_timer.cap = 0;
    return DLLM_OK;
}

DLLM_EXPORT unsigned long long dllm_launch_count(void) { return g_launches.load(); }

// ------------------------------------------------------------------ launch options
namespace dllm {
namespace {
std::atomic<int> g_pdl{1};
}
bool pdl_enabled() { return g_pdl.load(std::memory_order_relaxed) != 0; }
}  // namespace dllm

DLLM_EXPORT int dllm_set_pdl(int enable) {
    const int old = dllm::g_pdl.exchange(enable ? 1 : 0);
    return old;
}

// ------------------------------------------------------------------ allocation-free vocabulary step
DLLM_EXPORT int dllm_commit_entropy_noalloc(const float *logits, const uint8_t *valid, int B, int M,
                                            int V, float conf_thresh, float tau, int32_t *token,
                                            float *conf, float *entropy, float *max_entropy,
                                            int32_t *full_next, void *stream) {
    CHECK_ARG(max_entropy && full_next, "null pointer");
    CHECK_ARG(B > 0 && M >= 0 && V > 0, "sizes must be positive");
    CHECK_ARG(M <= 1024, "M must be <= 1024 (got %d)", M);
    if (M > 0) CHECK_ARG(logits && valid && token && conf && entropy, "null pointer");
    // every row needs at least one state, so B*M above the limit is rejected before the
    // int row count of the launch is formed
    if ((long long)B * M > commit_noalloc_max_states())
        return fail(DLLM_ERR_UNSUPPORTED,
                    "B*M = %lld rows exceed the allocation-free entry point's %d scratch states "
                    "(use dllm_commit_entropy with a workspace)",
                    (long long)B * M, commit_noalloc_max_states());
    const size_t states = commit_noalloc_states(B, M, V);
    if (states > (size_t)commit_noalloc_max_states())
        return fail(DLLM_ERR_UNSUPPORTED,
                    "B*M = %d rows need %zu scratch states; the allocation-free entry point holds %d "
                    "(use dllm_commit_entropy with a workspace)",
                    B * M, states, commit_noalloc_max_states());
    cudaStream_t st = as_stream(stream);
    Launch t(DLLM_KERNEL_VOCAB, st, 2);
    CHECK_CUDA(commit_entropy_noalloc(logits, valid, B, M, V, conf_thresh, tau, token, conf, entropy,
                                      max_entropy, full_next, st),
               "commit launch");
    return DLLM_OK;
}
