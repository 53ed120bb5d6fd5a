// front.cu -- the selection of a layer step fused with the gather of the selected rows
// (SPA-Cache, "1. Update identification via singular proxy", "2. Adaptive budget
// allocation" and the first stage of "3. Sparse execution"; EntropyCache, "How
// EntropyCache works", step 3).
//
// Grid (G, B): every CTA of sequence b computes the sequence's selection in shared
// memory (the same block-level selection as dllm_select_topk, so every CTA arrives at
// the same rows), CTA 0 of the sequence writes idx[b] and count[b], and CTA g then
// gathers rows g*R .. g*R+R-1 of the selection: RMSNorm(H[b, pos]) * gamma1 into Xn, the
// new proxy into the proxy cache, the rotary (cos, sin) of the position.  Selecting in
// every CTA costs a few microseconds of one block's work in parallel; it saves the launch
// of a separate gather kernel that would wait for the selection to finish.
//
// With the proxy projection's K-slice partials (bf16) or its proxies (fp32, one slice) as
// input, the kernel first computes the drift itself: CTA g of sequence b sums the partials
// and takes the cosine drift of rows g*N/G .. (g+1)*N/G-1 (one warp per row, the
// arithmetic of the cosine kernel), then the G
// CTAs of the sequence meet at a barrier (an arrival counter per sequence that the proxy
// projection zeroed; bounded wait) before they select.  The next kernel is released only
// after the barrier, so it cannot take the SM slots that the sequence's CTAs still need.
#include "cosine.cuh"
#include "rownorm.cuh"
#include "select.cuh"

namespace dllm {
namespace {
using namespace rownorm;

constexpr int kFT = 256;

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

template <class T>
__global__ void __launch_bounds__(kFT) k_select_gather(float *drift, const int32_t *__restrict__ forced, int F,
                                                       int k, float min_drift, int32_t *__restrict__ idx,
                                                       int32_t *__restrict__ count, int N, int k_max, int R,
                                                       const T *__restrict__ H, int d, const T *__restrict__ gamma,
                                                       float eps, T *__restrict__ Xn, float *proxy_cache,
                                                       float *proxy_cur, int r, const float *inv_freq,
                                                       int half_hd, float2 *rope_cs, DriftParts dp,
                                                       unsigned *status) {
    extern __shared__ uint32_t sm[];
    uint32_t *key = sm;                                                   // [N]
    int32_t *sel = reinterpret_cast<int32_t *>(key + N);                  // [N]
    uint8_t *flag = reinterpret_cast<uint8_t *>(sel + N);                 // [N]
    __shared__ float red[33];
    griddep_wait();
    const int b = blockIdx.y, g = blockIdx.x;
    if (dp.parts) {   // the drift of this CTA's share of the sequence's rows, then the barrier
        const int G = gridDim.x;
        const int n0 = (int)((long long)g * N / G), n1 = (int)((long long)(g + 1) * N / G);
        const long rows = (long)gridDim.y * N;
        const int lane = threadIdx.x & 31;
        for (int i = n0 + (threadIdx.x >> 5); i < n1; i += kFT / 32) {
            const long row = (long)b * N + i;
            const float dv = cosine_row<1>(dp.parts, dp.nparts, proxy_cache, proxy_cur, row, rows, r, lane);
            if (lane == 0) drift[row] = dv;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            atomicAdd(dp.arrive + b, 1u);
            const uint64_t t0 = globaltimer_ns();
            for (uint32_t it = 1; ld_acquire_u32(dp.arrive + b) < (unsigned)G; ++it) {
                if ((it & 255u) == 0 && globaltimer_ns() - t0 > kWaitLimitNs) {
                    raise_status(status, DLLM_STATUS_TIMEOUT);
                    break;
                }
            }
        }
        __syncthreads();
    }
    griddep_launch();
    const uint32_t total = select_sequence<kFT>(drift + (size_t)b * N, forced ? forced + (size_t)b * F : nullptr, F,
                                                k, min_drift, N, key, flag, sel);
    if (g == 0) {
        int32_t *row = idx + (size_t)b * N;
        for (int i = threadIdx.x; i < N; i += kFT) row[i] = sel[i];
        if (threadIdx.x == 0) {
            count[b] = (int32_t)total;
            if ((int)total > k_max) raise_status(status, DLLM_STATUS_COUNT_CLAMP);
        }
    }
    const int live = min((int)total, k_max);
    const int s1 = min(g * R + R, k_max);
    for (int s = g * R; s < s1; ++s) {
        const size_t m = (size_t)b * k_max + s;
        const int pos = s < live ? sel[s] : -1;
        if (rope_cs && threadIdx.x < half_hd) {
            float sn = 0.f, cs = 1.f;
            if (pos >= 0) sincosf((float)pos * inv_freq[threadIdx.x], &sn, &cs);
            rope_cs[m * half_hd + threadIdx.x] = make_float2(cs, sn);
        }
        T *out = Xn + m * d;
        if (pos < 0) {
            for (int e = threadIdx.x; e < d; e += kFT) out[e] = from_f32<T>(0.f);
            continue;
        }
        norm_row<T, T>(H + ((size_t)b * N + pos) * d, d, gamma, eps, out, red);
        if (proxy_cache && proxy_cur) {
            const size_t o = ((size_t)b * N + pos) * r;
            for (int e = threadIdx.x; e < r; e += kFT) proxy_cache[o + e] = __ldcg(proxy_cur + o + e);
        }
        __syncthreads();   // red[] is reused by the next row's norm
    }
}

}  // namespace

int select_gather_max_n() { return 4096; }

namespace {
// CTAs per sequence: about two CTAs per SM over all sequences' selected rows (R rows each)
int sg_ctas(int B, int k_max, int *R_out) {
    const long long rows = (long long)B * k_max;
    const long long target = 2LL * num_sms();
    int R = (int)((rows + target - 1) / target);
    if (R < 1) R = 1;
    *R_out = R;
    return (k_max + R - 1) / R;
}
}  // namespace

// The fused drift needs every CTA of a sequence resident at its barrier: the grid must
// fit the GPU at once (occupancy of the kernel at this shared-memory size, per device).
bool select_gather_fused_ok(int B, int N, int k_max, int dtype) {
    if (B <= 0 || N <= 0 || N > select_gather_max_n() || k_max <= 0) return false;
    int R = 1;
    const long long ctas = (long long)sg_ctas(B, k_max, &R) * B;
    struct Entry { int dev, dtype, smem, per_sm; };
    thread_local Entry cache[8] = {};
    thread_local int next = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    const int smem = N * 9;
    int per_sm = -1;
    for (const Entry &e : cache)
        if (e.per_sm > 0 && e.dev == dev && e.dtype == dtype && e.smem == smem) per_sm = e.per_sm;
    if (per_sm < 0) {
        cudaError_t err = dtype == DLLM_BF16
                              ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_select_gather<bf16>, kFT, smem)
                              : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_select_gather<float>, kFT, smem);
        if (err != cudaSuccess || per_sm <= 0) {
            (void)cudaGetLastError();
            return false;
        }
        cache[next] = Entry{dev, dtype, smem, per_sm};
        next = (next + 1) % 8;
    }
    return ctas <= (long long)per_sm * num_sms();
}

template <class T>
cudaError_t select_gather(float *drift, const int32_t *forced, int F, int k, float min_drift, int32_t *idx,
                          int32_t *count, int B, int N, int k_max, const T *H, int d, const T *gamma, float eps,
                          T *Xn, float *proxy_cache, float *proxy_cur, int r, const float *inv_freq,
                          int half_hd, float2 *rope_cs, DriftParts dp, unsigned *status, cudaStream_t st) {
    if (B <= 0 || N <= 0 || k_max <= 0) return cudaSuccess;
    if (N > select_gather_max_n()) return cudaErrorInvalidValue;
    if (dp.parts && (r > 128 || r % 32 || !proxy_cache || !proxy_cur || !dp.arrive)) return cudaErrorInvalidValue;
    int R = 1;
    const int G = sg_ctas(B, k_max, &R);
    if (dp.parts && !select_gather_fused_ok(B, N, k_max, sizeof(T) == 2 ? DLLM_BF16 : DLLM_F32))
        return cudaErrorInvalidValue;
    const size_t smem = (size_t)N * 9;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k_select_gather<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_kernel(k_select_gather<T>, dim3(G, B), dim3(kFT), smem, st, 1, drift, forced, F, k, min_drift,
                         idx, count, N, k_max, R, H, d, gamma, eps, Xn, proxy_cache, proxy_cur, r, inv_freq,
                         half_hd, rope_cs, dp, status);
}

template cudaError_t select_gather<bf16>(float *, const int32_t *, int, int, float, int32_t *, int32_t *, int, int,
                                         int, const bf16 *, int, const bf16 *, float, bf16 *, float *, float *, int,
                                         const float *, int, float2 *, DriftParts, unsigned *, cudaStream_t);
template cudaError_t select_gather<float>(float *, const int32_t *, int, int, float, int32_t *, int32_t *, int, int,
                                          int, const float *, int, const float *, float, float *, float *, float *,
                                          int, const float *, int, float2 *, DriftParts, unsigned *, cudaStream_t);

}  // namespace dllm
