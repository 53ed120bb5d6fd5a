// cluster.cu -- cluster-granular proxy ("Polestar: drift-aware cache correction and token
// commit", 2. A, Polestar-Cache: local window and clustering, sparse updates).  The window's
// hidden states are clustered with spherical k-means, the residuals of each row against its
// centroid direction are quantised to NVFP4, and each step the clusters whose centroid
// direction drifted most are refreshed: their member rows form the selection.
//
//   k-means (Lloyd): a_i = argmax_k <x_i, c_k> (unit centroids; lowest k on ties),
//     c_k = normalise(sum_{a_i = k} x_i / |x_i|) summed in row order (deterministic), an
//     empty cluster keeping its centroid;
//   residual r_i = x_i - |x_i| c_{a_i};
//   NVFP4: per 16-element block s_b = E4M3(amax / (6 g)), codes E2M1(x / (s_b g)), both by
//     the sm_103a conversions (round to nearest even, saturating); two codes per byte,
//     element 2j in the low nibble;
//   cluster drift d_k = 1 - cos(c_k^t, c_k^{t-1}); the kc largest (lower k on ties) are
//     chosen and their member rows listed ascending.
#include <math.h>

#include "internal.h"

namespace dllm {
namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Block-wide sum over blockDim.x threads (a multiple of 32, <= 1024); every thread gets it.
__device__ float block_sum(float v, float *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v = warp_sum(v);
    __syncthreads();   // red may still be read from a previous call
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.f;
    for (int w = 0; w < nw; ++w) t += red[w];   // same order in every thread
    return t;
}

// Rows of C [rows, D] scaled to unit length (a zero row stays zero).  One CTA per row.
__global__ void __launch_bounds__(256) k_normalize_rows(float *__restrict__ C, int D) {
    __shared__ float red[32];
    griddep_wait();
    griddep_launch();
    float *c = C + (size_t)blockIdx.x * D;
    float ss = 0.f;
    for (int d = threadIdx.x; d < D; d += blockDim.x) ss = fmaf(c[d], c[d], ss);
    const float n2 = block_sum(ss, red);
    if (n2 > 0.f) {
        const float inv = 1.f / sqrtf(n2);
        for (int d = threadIdx.x; d < D; d += blockDim.x) c[d] *= inv;
    }
}

// One CTA per row: the row staged in shared memory (16-byte loads), |x_i|, and
// argmax_k <x_i, c_k> with the clusters dealt to the warps (lowest k on ties).
constexpr int kAsgThreads = 256;
constexpr int kMaxK = 256;

__global__ void __launch_bounds__(kAsgThreads)
    k_kmeans_assign(const float *__restrict__ X, const float *__restrict__ C, int32_t *__restrict__ assign,
                    float *__restrict__ xnorm, int N, int D, int K) {
    extern __shared__ float4 xs4[];   // [D / 4]
    __shared__ float dots[kMaxK];
    __shared__ float red[32];
    griddep_wait();
    griddep_launch();
    const long row = blockIdx.x;
    const int b = (int)(row / N), lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int D4 = D / 4;
    const float4 *x4 = reinterpret_cast<const float4 *>(X + row * D);
    float ss = 0.f;
    for (int j = threadIdx.x; j < D4; j += kAsgThreads) {
        const float4 v = x4[j];
        xs4[j] = v;
        ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
    }
    const float n2 = block_sum(ss, red);   // also publishes the staged row
    for (int k = warp; k < K; k += kAsgThreads / 32) {
        const float4 *c4 = reinterpret_cast<const float4 *>(C + ((size_t)b * K + k) * D);
        float dot = 0.f;
#pragma unroll 4
        for (int j = lane; j < D4; j += 32) {
            const float4 c = c4[j], v = xs4[j];
            dot = fmaf(v.x, c.x, fmaf(v.y, c.y, fmaf(v.z, c.z, fmaf(v.w, c.w, dot))));
        }
        dot = warp_sum(dot);
        if (lane == 0) dots[k] = dot;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int best = 0;
        for (int k = 1; k < K; ++k)
            if (dots[k] > dots[best]) best = k;   // strict: the lowest k keeps a tie
        assign[row] = best;
        xnorm[row] = sqrtf(n2);
    }
}

// One CTA per (sequence, cluster): c_k = normalise(sum over member rows, in row order, of
// x_i / |x_i|); unchanged when the sum is zero.  Per chunk of 1024 rows the members are
// compacted in row order into shared memory (block scan), then summed four at a time (their
// loads in flight together); each thread keeps the sums of its dimensions d = tid + 256 j
// in registers.
constexpr int kUpdThreads = 256;
constexpr int kUpdDims = 32;   // dimensions per thread: D <= 8192
constexpr int kUpdChunk = 1024;

__global__ void __launch_bounds__(kUpdThreads)
    k_kmeans_update(const float *__restrict__ X, const int32_t *__restrict__ assign,
                    const float *__restrict__ xnorm, float *__restrict__ C, int N, int D, int K) {
    __shared__ int mem_s[kUpdChunk];
    __shared__ float inv_s[kUpdChunk];
    __shared__ int wsum[33];
    __shared__ float red[32];
    griddep_wait();
    griddep_launch();
    const int b = blockIdx.y, k = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int kPer = kUpdChunk / kUpdThreads;   // rows per thread in a chunk (contiguous)
    float acc[kUpdDims];
#pragma unroll
    for (int j = 0; j < kUpdDims; ++j) acc[j] = 0.f;
    for (int c0 = 0; c0 < N; c0 += kUpdChunk) {
        // members of this chunk, in row order
        int mine = 0;
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int i = c0 + tid * kPer + q;
            mine += i < N && assign[(size_t)b * N + i] == k && xnorm[(size_t)b * N + i] > 0.f;
        }
        int incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        __syncthreads();   // the previous chunk's list has been read
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int w = lane < kUpdThreads / 32 ? wsum[lane] : 0;
            int sc = w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, sc, o);
                if (lane >= o) sc += y;
            }
            wsum[lane] = sc - w;
            if (lane == 31) wsum[32] = sc;
        }
        __syncthreads();
        int pos = wsum[warp] + incl - mine;
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
            const int i = c0 + tid * kPer + q;
            if (i < N && assign[(size_t)b * N + i] == k && xnorm[(size_t)b * N + i] > 0.f) {
                mem_s[pos] = i;
                inv_s[pos] = 1.f / xnorm[(size_t)b * N + i];
                ++pos;
            }
        }
        __syncthreads();
        const int nm = wsum[32];
        for (int m = 0; m < nm; m += 4) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (m + u < nm) {
                    const float inv = inv_s[m + u];
                    const float *x = X + ((size_t)b * N + mem_s[m + u]) * D;
#pragma unroll
                    for (int j = 0; j < kUpdDims; ++j) {
                        const int d = tid + kUpdThreads * j;
                        if (d < D) acc[j] = fmaf(x[d], inv, acc[j]);
                    }
                }
            }
        }
    }
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < kUpdDims; ++j) ss = fmaf(acc[j], acc[j], ss);
    const float n2 = block_sum(ss, red);
    if (n2 > 0.f) {
        const float inv = 1.f / sqrtf(n2);
        float *c = C + ((size_t)b * K + k) * D;
#pragma unroll
        for (int j = 0; j < kUpdDims; ++j) {
            const int d = tid + kUpdThreads * j;
            if (d < D) c[d] = acc[j] * inv;
        }
    }
}

// R = x_i - |x_i| c_{a_i}, elementwise.
__global__ void __launch_bounds__(256)
    k_cluster_residual(const float *__restrict__ X, const float *__restrict__ C, const int32_t *__restrict__ assign,
                       const float *__restrict__ xnorm, float *__restrict__ R, int N, int D, int K, long total) {
    griddep_wait();
    griddep_launch();
    const long t = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= total) return;
    const long row = t / D;
    const int d = (int)(t - row * D);
    const int b = (int)(row / N);
    const int a = assign[row];
    if (a < 0 || a >= K) {   // no cluster: the whole row is residual
        R[t] = X[t];
        return;
    }
    const float *c = C + ((size_t)b * K + a) * D;
    R[t] = X[t] - xnorm[row] * c[d];
}

__device__ __forceinline__ uint32_t e2m1x8(const float *q) {   // q[0] -> low nibble of byte 0
    uint32_t out;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(out)
        : "f"(q[0]), "f"(q[1]), "f"(q[2]), "f"(q[3]), "f"(q[4]), "f"(q[5]), "f"(q[6]), "f"(q[7]));
    return out;
}

// One thread per 16-element block: E4M3 block scale, then 16 E2M1 codes in 8 bytes.
__global__ void __launch_bounds__(256)
    k_nvfp4_quant(const float *__restrict__ R, float g, uint8_t *__restrict__ codes, uint8_t *__restrict__ scales,
                  long blocks) {
    griddep_wait();
    griddep_launch();
    const long t = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= blocks) return;
    float v[16];
    const float4 *src = reinterpret_cast<const float4 *>(R + t * 16);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float4 f = src[j];
        v[4 * j] = f.x;
        v[4 * j + 1] = f.y;
        v[4 * j + 2] = f.z;
        v[4 * j + 3] = f.w;
    }
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
    const float s_in = amax / (6.f * g);
    unsigned short s2;   // low byte: E4M3 of s_in
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(s2) : "f"(0.f), "f"(s_in));
    unsigned h2;         // the scale back as f16 (exact), low half
    asm("{\n\t.reg .b16 lo;\n\tmov.b16 lo, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}" : "=r"(h2) : "h"(s2));
    const float s_val = __half2float(__ushort_as_half((unsigned short)(h2 & 0xffffu)));
    const float denom = s_val * g;
    uint2 out = make_uint2(0u, 0u);
    if (denom > 0.f) {
        float q[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) q[j] = v[j] / denom;
        out.x = e2m1x8(q);
        out.y = e2m1x8(q + 8);
    }
    *reinterpret_cast<uint2 *>(codes + t * 8) = out;
    scales[t] = (uint8_t)(s2 & 0xffu);
}

// One thread per 16-element block: value = E2M1(code) * E4M3(scale) * g.  The first product
// is exact in fp32 (2 + 4 significant bits), so each value is rounded once, by * g.
__global__ void __launch_bounds__(256)
    k_nvfp4_dequant(const uint8_t *__restrict__ codes, const uint8_t *__restrict__ scales, float g,
                    float *__restrict__ out, long blocks) {
    griddep_wait();
    griddep_launch();
    const long t = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= blocks) return;
    unsigned h2;
    asm("{\n\t.reg .b16 lo;\n\tmov.b16 lo, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
        : "=r"(h2)
        : "h"((unsigned short)scales[t]));
    const float s = __half2float(__ushort_as_half((unsigned short)(h2 & 0xffffu)));
    const uint2 q = *reinterpret_cast<const uint2 *>(codes + t * 8);
    float v[16];
#pragma unroll
    for (int w = 0; w < 2; ++w) {
        const uint32_t word = w == 0 ? q.x : q.y;
#pragma unroll
        for (int by = 0; by < 4; ++by) {
            unsigned pair;   // two codes of one byte -> f16x2 (low nibble -> low half)
            asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}"
                : "=r"(pair)
                : "r"((word >> (8 * by)) & 0xffu));
            v[w * 8 + by * 2] = __half2float(__ushort_as_half((unsigned short)(pair & 0xffffu))) * s * g;
            v[w * 8 + by * 2 + 1] = __half2float(__ushort_as_half((unsigned short)(pair >> 16))) * s * g;
        }
    }
    float4 *dst = reinterpret_cast<float4 *>(out + t * 16);
#pragma unroll
    for (int j = 0; j < 4; ++j) dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
}

// One CTA per sequence: cluster drifts, the kc largest, their member rows ascending.
constexpr int kSelThreads = 256;
constexpr int kMaxClusters = 256;

__global__ void __launch_bounds__(kSelThreads)
    k_cluster_select(const float *__restrict__ Cn, const float *__restrict__ Cp, const int32_t *__restrict__ assign,
                     int kc, int32_t *__restrict__ idx, int32_t *__restrict__ count, int N, int D, int K) {
    __shared__ float drift[kMaxClusters];
    __shared__ uint8_t chosen[kMaxClusters];
    __shared__ int wsum[33];
    griddep_wait();
    griddep_launch();
    const int b = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int k = warp; k < K; k += kSelThreads / 32) {
        const float *a = Cn + ((size_t)b * K + k) * D;
        const float *p = Cp + ((size_t)b * K + k) * D;
        float dot = 0.f, na = 0.f, nb = 0.f;
#pragma unroll 8
        for (int d = lane; d < D; d += 32) {
            dot = fmaf(a[d], p[d], dot);
            na = fmaf(a[d], a[d], na);
            nb = fmaf(p[d], p[d], nb);
        }
        dot = warp_sum(dot);
        na = warp_sum(na);
        nb = warp_sum(nb);
        if (lane == 0) {
            float dr;
            if (na > 0.f && nb > 0.f) dr = fminf(fmaxf(1.f - dot / sqrtf(na * nb), 0.f), 2.f);
            else dr = (na > 0.f) != (nb > 0.f) ? 1.f : 0.f;
            drift[k] = dr;
        }
    }
    __syncthreads();
    for (int k = threadIdx.x; k < K; k += kSelThreads) {
        int rank = 0;
        for (int j = 0; j < K; ++j) rank += drift[j] > drift[k] || (drift[j] == drift[k] && j < k);
        chosen[k] = rank < kc;
    }
    __syncthreads();
    // member rows in ascending order: contiguous chunk per thread, block scan of the counts
    const int C_ = (N + kSelThreads - 1) / kSelThreads;
    const int i0 = min(N, (int)threadIdx.x * C_), i1 = min(N, i0 + C_);
    const int32_t *a = assign + (size_t)b * N;
    int n = 0;
    for (int i = i0; i < i1; ++i) n += (unsigned)a[i] < (unsigned)K && chosen[a[i]];
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int w = lane < kSelThreads / 32 ? wsum[lane] : 0;
        int s = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        wsum[lane] = s - w;
        if (lane == 31) wsum[32] = s;
    }
    __syncthreads();
    int out = wsum[warp] + incl - n;
    int32_t *row = idx + (size_t)b * N;
    for (int i = i0; i < i1; ++i)
        if ((unsigned)a[i] < (unsigned)K && chosen[a[i]]) row[out++] = i;
    const int total = wsum[32];
    for (int i = total + (int)threadIdx.x; i < N; i += kSelThreads) row[i] = -1;
    if (threadIdx.x == 0) count[b] = total;
}

}  // namespace

cudaError_t spherical_kmeans(const float *X, float *C, int32_t *assign, float *xnorm, int B, int N, int D, int K,
                             int iters, cudaStream_t st) {
    if (B <= 0 || N <= 0) return cudaSuccess;
    if (D <= 0 || D % 4 || K <= 0 || K > kMaxK || D > kUpdThreads * kUpdDims) return cudaErrorInvalidValue;
    cudaError_t e = launch_kernel(k_normalize_rows, dim3((unsigned)(B * K)), dim3(256), 0, st, 1, C, D);
    const long rows = (long)B * N;
    const dim3 ag((unsigned)rows);
    const size_t xs = (size_t)D * 4;   // the staged row (<= 32 KB)
    for (int it = 0; e == cudaSuccess && it < iters; ++it) {
        e = launch_kernel(k_kmeans_assign, ag, dim3(kAsgThreads), xs, st, 1, X, (const float *)C, assign, xnorm, N,
                          D, K);
        if (e == cudaSuccess)
            e = launch_kernel(k_kmeans_update, dim3((unsigned)K, (unsigned)B), dim3(kUpdThreads), 0, st, 1, X,
                              (const int32_t *)assign, (const float *)xnorm, C, N, D, K);
    }
    if (e == cudaSuccess)
        e = launch_kernel(k_kmeans_assign, ag, dim3(kAsgThreads), xs, st, 1, X, (const float *)C, assign, xnorm, N,
                          D, K);
    return e;
}

cudaError_t cluster_residual(const float *X, const float *C, const int32_t *assign, const float *xnorm, float *R,
                             int B, int N, int D, int K, cudaStream_t st) {
    const long total = (long)B * N * D;
    if (total <= 0) return cudaSuccess;
    return launch_kernel(k_cluster_residual, dim3((unsigned)((total + 255) / 256)), dim3(256), 0, st, 1, X, C,
                         assign, xnorm, R, N, D, K, total);
}

cudaError_t nvfp4_quantize(const float *R, float g, uint8_t *codes, uint8_t *scales, long rows, int D,
                           cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    if (D <= 0 || D % 16) return cudaErrorInvalidValue;
    const long blocks = rows * (D / 16);
    return launch_kernel(k_nvfp4_quant, dim3((unsigned)((blocks + 255) / 256)), dim3(256), 0, st, 1, R, g, codes,
                         scales, blocks);
}

cudaError_t nvfp4_dequantize(const uint8_t *codes, const uint8_t *scales, float g, float *out, long rows, int D,
                             cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    if (D <= 0 || D % 16) return cudaErrorInvalidValue;
    const long blocks = rows * (D / 16);
    return launch_kernel(k_nvfp4_dequant, dim3((unsigned)((blocks + 255) / 256)), dim3(256), 0, st, 1, codes, scales,
                         g, out, blocks);
}

cudaError_t cluster_select(const float *Cn, const float *Cp, const int32_t *assign, int kc, int32_t *idx,
                           int32_t *count, int B, int N, int D, int K, cudaStream_t st) {
    if (B <= 0 || N <= 0) return cudaSuccess;
    if (K <= 0 || K > kMaxClusters) return cudaErrorInvalidValue;
    return launch_kernel(k_cluster_select, dim3((unsigned)B), dim3(kSelThreads), 0, st, 1, Cn, Cp, assign, kc, idx,
                         count, N, D, K);
}

}  // namespace dllm
