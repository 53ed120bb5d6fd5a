// rowops.cu -- per-row kernels of the refresh (SPA-Cache, "1. Update identification
// via singular proxy" and "3. Sparse execution"): gather + RMSNorm of the selected
// rows, RMSNorm of the attention residual, the cosine drift score, and the one-time
// weight packing.  All of them are memory-bound row sweeps: one CTA (or warp) per
// row, coalesced loads, shuffle reductions.
#include "cosine.cuh"
#include "rownorm.cuh"

namespace dllm {
namespace {
using namespace rownorm;

// Xn[m] = RMSNorm(H[b, pos]) * gamma1 for the live selected rows, zeros otherwise;
// proxy_cache[b, pos] <- proxy_cur[b, pos];  rope_cs[m, i] = (cos, sin) of the rotary
// angle pos * inv_freq[i] (fp32), used by the QKV epilogue.
template <class T>
__global__ void __launch_bounds__(256) k_gather_rmsnorm(const T *__restrict__ H, SelRows sel, int d,
                                                        const T *__restrict__ gamma, float eps,
                                                        T *__restrict__ Xn, float *proxy_cache,
                                                        const float *proxy_cur, int r,
                                                        const float *inv_freq, int half_hd,
                                                        float2 *rope_cs, unsigned *status) {
    __shared__ float red[33];
    griddep_wait();
    griddep_launch();
    const int m = blockIdx.x;
    int b, pos;
    sel.locate(m, b, pos);
    if (threadIdx.x == 0 && m % sel.k_max == 0 && sel.count[b] > sel.k_max)
        raise_status(status, DLLM_STATUS_COUNT_CLAMP);
    if (rope_cs && threadIdx.x < half_hd) {
        float sn = 0.f, cs = 1.f;
        if (pos >= 0) sincosf((float)pos * inv_freq[threadIdx.x], &sn, &cs);
        rope_cs[(size_t)m * half_hd + threadIdx.x] = make_float2(cs, sn);
    }
    T *out = Xn + (size_t)m * d;
    if (pos < 0) {
        for (int e = threadIdx.x; e < d; e += 256) out[e] = from_f32<T>(0.f);
        return;
    }
    const T *row = H + ((size_t)b * sel.N + pos) * d;
    norm_row<T, T>(row, d, gamma, eps, out, red);
    if (proxy_cache && proxy_cur) {
        const size_t o = ((size_t)b * sel.N + pos) * r;
        for (int e = threadIdx.x; e < r; e += 256) proxy_cache[o + e] = proxy_cur[o + e];
    }
}

// Xn2[m] = RMSNorm(h1[m]) * gamma2 (h1 in fp32).
template <class T>
__global__ void __launch_bounds__(256) k_rmsnorm_rows(const float *__restrict__ h1, int d,
                                                      const T *__restrict__ gamma, float eps,
                                                      T *__restrict__ Xn2) {
    __shared__ float red[33];
    griddep_wait();
    griddep_launch();
    norm_row<float, T>(h1 + (size_t)blockIdx.x * d, d, gamma, eps, Xn2 + (size_t)blockIdx.x * d, red);
}

// The cosine drift of every row (cosine.cuh), one warp per row: r <= 128 keeps one float4
// chunk per lane, wider proxies (r <= 1024) up to eight.
template <int MAXCH>
__global__ void __launch_bounds__(256) k_cosine_drift(const float *__restrict__ parts, int nparts,
                                                      const float *__restrict__ cached,
                                                      float *__restrict__ cur,
                                                      float *__restrict__ drift, long rows, int r) {
    griddep_wait();
    griddep_launch();
    const long row = (long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const float out = cosine_row<MAXCH>(parts, nparts, cached, cur, row, rows, r, lane);
    if (lane == 0) drift[row] = out;
}

// dst row (head h, p) = src row (head h, p even ? p/2 : p/2 + hd/2): rotary pairs adjacent.
template <class T>
__global__ void k_pack_rope(const T *__restrict__ src, T *__restrict__ dst, int cols, int hd) {
    const int row = blockIdx.x;
    const int h = row / hd, p = row - h * hd;
    const int srow = h * hd + ((p & 1) ? (p >> 1) + hd / 2 : (p >> 1));
    for (int e = threadIdx.x; e < cols; e += blockDim.x) dst[(size_t)row * cols + e] = src[(size_t)srow * cols + e];
}

// dst row 2j = a row j, dst row 2j+1 = b row j.
template <class T>
__global__ void k_pack_interleave(const T *__restrict__ a, const T *__restrict__ b,
                                  T *__restrict__ dst, int cols) {
    const int row = blockIdx.x;
    const T *s = (row & 1) ? b : a;
    const int j = row >> 1;
    for (int e = threadIdx.x; e < cols; e += blockDim.x) dst[(size_t)row * cols + e] = s[(size_t)j * cols + e];
}

__global__ void k_rope_inv_freq(float *dst, int hd, float theta) {
    const int i = threadIdx.x;
    if (i < hd / 2) dst[i] = (float)pow((double)theta, -2.0 * (double)i / (double)hd);
}

}  // namespace

template <class T>
cudaError_t gather_rmsnorm(const T *H, SelRows sel, int B, int d, const T *gamma, float eps, T *Xn,
                           float *proxy_cache, const float *proxy_cur, int r, const float *inv_freq,
                           int half_hd, float2 *rope_cs, unsigned *status, cudaStream_t st) {
    const int M = B * sel.k_max;
    if (M <= 0) return cudaSuccess;
    return launch_kernel(k_gather_rmsnorm<T>, dim3(M), dim3(256), 0, st, 1, H, sel, d, gamma, eps, Xn,
                         proxy_cache, proxy_cur, r, inv_freq, half_hd, rope_cs, status);
}

template <class T>
cudaError_t rmsnorm_rows(const float *h1, int M, int d, const T *gamma, float eps, T *Xn2,
                         cudaStream_t st) {
    if (M <= 0) return cudaSuccess;
    return launch_kernel(k_rmsnorm_rows<T>, dim3(M), dim3(256), 0, st, 1, h1, d, gamma, eps, Xn2);
    return cudaGetLastError();
}

cudaError_t cosine_drift(const float *parts, int nparts, const float *cached, float *cur,
                         float *drift, long rows, int r, cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    if (r <= 128)
        return launch_kernel(k_cosine_drift<1>, dim3((unsigned)((rows + 7) / 8)), dim3(256), 0, st, 1, parts,
                             nparts, cached, cur, drift, rows, r);
    return launch_kernel(k_cosine_drift<8>, dim3((unsigned)((rows + 7) / 8)), dim3(256), 0, st, 1, parts,
                         nparts, cached, cur, drift, rows, r);
}

template <class T>
cudaError_t pack_rows_rope(const T *src, T *dst, int rows, int cols, int hd, cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    (void)cudaGetLastError();   // a stale error of an earlier, already reported call is not this launch's
    k_pack_rope<T><<<rows, 256, 0, st>>>(src, dst, cols, hd);
    return cudaGetLastError();
}

template <class T>
cudaError_t pack_rows_interleave(const T *a, const T *b, T *dst, int rows, int cols, cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    (void)cudaGetLastError();
    k_pack_interleave<T><<<2 * rows, 256, 0, st>>>(a, b, dst, cols);
    return cudaGetLastError();
}

cudaError_t rope_inv_freq(float *dst, int hd, float theta, cudaStream_t st) {
    (void)cudaGetLastError();
    k_rope_inv_freq<<<1, 128, 0, st>>>(dst, hd, theta);
    return cudaGetLastError();
}

#define DLLM_ROWOPS(T)                                                                           \
    template cudaError_t gather_rmsnorm<T>(const T *, SelRows, int, int, const T *, float, T *,  \
                                           float *, const float *, int, const float *, int, float2 *,   \
                                           unsigned *, cudaStream_t);                                   \
    template cudaError_t rmsnorm_rows<T>(const float *, int, int, const T *, float, T *,         \
                                         cudaStream_t);                                          \
    template cudaError_t pack_rows_rope<T>(const T *, T *, int, int, int, cudaStream_t);         \
    template cudaError_t pack_rows_interleave<T>(const T *, const T *, T *, int, int, cudaStream_t);
DLLM_ROWOPS(float)
DLLM_ROWOPS(bf16)
#undef DLLM_ROWOPS

}  // namespace dllm

// ---------------------------------------------------------------------------
// Token embedding lookup and the final RMSNorm of chosen rows (decode loop around
// the refresh: the inputs of layer 0 and the rows fed to the LM head).
namespace dllm {
namespace {
using namespace rownorm;

template <class T>
__global__ void __launch_bounds__(256) k_embed(const T *__restrict__ E, const int32_t *__restrict__ tokens,
                                               const int32_t *__restrict__ rows, int R, T *__restrict__ H,
                                               int N, int d, int V) {
    griddep_wait();
    griddep_launch();
    const int b = blockIdx.y;
    int i = blockIdx.x;
    if (rows) {
        i = rows[(size_t)b * R + blockIdx.x];
        if (i < 0 || i >= N) return;
    }
    const int tok = tokens[(size_t)b * N + i];
    T *dst = H + ((size_t)b * N + i) * d;
    if (tok < 0 || tok >= V) {
        for (int e = threadIdx.x; e < d; e += 256) dst[e] = from_f32<T>(0.f);
        return;
    }
    const T *src = E + (size_t)tok * d;
    for (int e = threadIdx.x; e < d; e += 256) dst[e] = src[e];
}

template <class T>
__global__ void __launch_bounds__(256) k_rows_rmsnorm(const T *__restrict__ H, const int32_t *__restrict__ rows,
                                                      int R, const T *__restrict__ gamma, float eps,
                                                      T *__restrict__ out, int N, int d) {
    __shared__ float red[33];
    griddep_wait();
    griddep_launch();
    const int b = blockIdx.y, j = blockIdx.x;
    const int i = rows[(size_t)b * R + j];
    T *o = out + ((size_t)b * R + j) * d;
    if (i < 0 || i >= N) {
        for (int e = threadIdx.x; e < d; e += 256) o[e] = from_f32<T>(0.f);
        return;
    }
    const T *row = H + ((size_t)b * N + i) * d;
    float ss = 0.f;
    for (int e = threadIdx.x; e < d; e += 256) {
        const float x = to_f32<T>(row[e]);
        ss = fmaf(x, x, ss);
    }
    ss = block_sum<256>(ss, red);
    const float inv = 1.0f / sqrtf(ss / (float)d + eps);
    for (int e = threadIdx.x; e < d; e += 256) o[e] = from_f32<T>(to_f32<T>(row[e]) * inv * to_f32<T>(gamma[e]));
}

// One CTA per packed row: 16-byte copies of the selected cache row, or zeros.
// dst_t[m] = src_t[b, pos] for each of the caches t = blockIdx.y that share one selection
// (zeros for rows that are not live).
__global__ void __launch_bounds__(128) k_gather_rows(GatherSet gs, SelRows sel) {
    griddep_wait();
    griddep_launch();
    const int m = blockIdx.x, t = blockIdx.y;
    const int vecs = gs.vecs[t];
    int b, pos;
    sel.locate(m, b, pos);
    uint4 *o = static_cast<uint4 *>(gs.dst[t]) + (size_t)m * vecs;
    if (pos < 0) {
        for (int v = threadIdx.x; v < vecs; v += 128) o[v] = make_uint4(0u, 0u, 0u, 0u);
        return;
    }
    const uint4 *row = static_cast<const uint4 *>(gs.src[t]) + ((size_t)b * sel.N + pos) * vecs;
    for (int v = threadIdx.x; v < vecs; v += 128) o[v] = row[v];
}

}  // namespace

cudaError_t gather_rows(const GatherSet &gs, int n, SelRows sel, int B, cudaStream_t st) {
    const long M = (long)B * sel.k_max;
    if (M <= 0 || n <= 0) return cudaSuccess;
    if (n > kGatherMax) return cudaErrorInvalidValue;
    return launch_kernel(k_gather_rows, dim3((unsigned)M, (unsigned)n), dim3(128), 0, st, 1, gs, sel);
}

template <class T>
cudaError_t embed_rows(const T *E, const int32_t *tokens, const int32_t *rows, int R, T *H, int B,
                       int N, int d, int V, cudaStream_t st) {
    const int nr = rows ? R : N;
    if (B <= 0 || nr <= 0) return cudaSuccess;
    return launch_kernel(k_embed<T>, dim3(nr, B), dim3(256), 0, st, 1, E, tokens, rows, R, H, N, d, V);
    return cudaGetLastError();
}

template <class T>
cudaError_t rows_rmsnorm(const T *H, const int32_t *rows, int R, const T *gamma, float eps, T *out,
                         int B, int N, int d, cudaStream_t st) {
    if (B <= 0 || R <= 0) return cudaSuccess;
    return launch_kernel(k_rows_rmsnorm<T>, dim3(R, B), dim3(256), 0, st, 1, H, rows, R, gamma, eps, out, N, d);
    return cudaGetLastError();
}

template cudaError_t embed_rows<float>(const float *, const int32_t *, const int32_t *, int, float *, int, int, int, int, cudaStream_t);
template cudaError_t embed_rows<bf16>(const bf16 *, const int32_t *, const int32_t *, int, bf16 *, int, int, int, int, cudaStream_t);
template cudaError_t rows_rmsnorm<float>(const float *, const int32_t *, int, const float *, float, float *, int, int, int, cudaStream_t);
template cudaError_t rows_rmsnorm<bf16>(const bf16 *, const int32_t *, int, const bf16 *, float, bf16 *, int, int, int, cudaStream_t);

}  // namespace dllm
