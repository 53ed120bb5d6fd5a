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
#include "rownorm.cuh"
#include "select.cuh"

namespace dllm {
namespace {
using namespace rownorm;

constexpr int kFT = 256;

template <class T>
__global__ void __launch_bounds__(kFT) k_select_gather(const float *__restrict__ drift,
                                                       const int32_t *__restrict__ forced, int F, int k,
                                                       float min_drift, int32_t *__restrict__ idx,
                                                       int32_t *__restrict__ count, int N, int k_max, int R,
                                                       const T *__restrict__ H, int d, const T *__restrict__ gamma,
                                                       float eps, T *__restrict__ Xn, float *proxy_cache,
                                                       const float *proxy_cur, int r, const float *inv_freq,
                                                       int half_hd, float2 *rope_cs, unsigned *status) {
    extern __shared__ uint32_t sm[];
    uint32_t *key = sm;                                                   // [N]
    int32_t *sel = reinterpret_cast<int32_t *>(key + N);                  // [N]
    uint8_t *flag = reinterpret_cast<uint8_t *>(sel + N);                 // [N]
    __shared__ float red[33];
    griddep_wait();
    griddep_launch();
    const int b = blockIdx.y, g = blockIdx.x;
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
            for (int e = threadIdx.x; e < r; e += kFT) proxy_cache[o + e] = proxy_cur[o + e];
        }
        __syncthreads();   // red[] is reused by the next row's norm
    }
}

}  // namespace

int select_gather_max_n() { return 4096; }

template <class T>
cudaError_t select_gather(const float *drift, const int32_t *forced, int F, int k, float min_drift, int32_t *idx,
                          int32_t *count, int B, int N, int k_max, const T *H, int d, const T *gamma, float eps,
                          T *Xn, float *proxy_cache, const float *proxy_cur, int r, const float *inv_freq,
                          int half_hd, float2 *rope_cs, unsigned *status, cudaStream_t st) {
    if (B <= 0 || N <= 0 || k_max <= 0) return cudaSuccess;
    if (N > select_gather_max_n()) return cudaErrorInvalidValue;
    // rows per CTA: about two CTAs per SM over all sequences
    const long long rows = (long long)B * k_max;
    const long long target = 2LL * num_sms();
    int R = (int)((rows + target - 1) / target);
    if (R < 1) R = 1;
    const int G = (k_max + R - 1) / R;
    const size_t smem = (size_t)N * 9;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k_select_gather<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch_kernel(k_select_gather<T>, dim3(G, B), dim3(kFT), smem, st, 1, drift, forced, F, k, min_drift,
                         idx, count, N, k_max, R, H, d, gamma, eps, Xn, proxy_cache, proxy_cur, r, inv_freq,
                         half_hd, rope_cs, status);
}

template cudaError_t select_gather<bf16>(const float *, const int32_t *, int, int, float, int32_t *, int32_t *, int,
                                         int, int, const bf16 *, int, const bf16 *, float, bf16 *, float *,
                                         const float *, int, const float *, int, float2 *, unsigned *, cudaStream_t);
template cudaError_t select_gather<float>(const float *, const int32_t *, int, int, float, int32_t *, int32_t *, int,
                                          int, int, const float *, int, const float *, float, float *, float *,
                                          const float *, int, const float *, int, float2 *, unsigned *,
                                          cudaStream_t);

}  // namespace dllm
