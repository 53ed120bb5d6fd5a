// attention_simt.cu -- non-causal attention of the selected queries over the whole
// (partially refreshed) cache on the CUDA cores (SPA-Cache, "3. Sparse execution").
// Used for the fp32 configuration.
//
// One CTA (4 warps) per (query row, head); warp w takes a quarter of the keys.  Each lane
// holds hd/32 dims of the query (pre-scaled), so a key's score is a warp all-reduce over
// one coalesced key row; two keys go through each step so that their reductions and
// exponentials overlap.  Each warp keeps the streaming (running max / running sum) form in
// fp32; the four warps' states are merged through shared memory at the end, in warp order.
#include "internal.h"

namespace dllm {
namespace {

constexpr int kWarpsA = 4;

template <class T, int EPL>
__global__ void __launch_bounds__(kWarpsA * 32) k_attention_simt(const T *__restrict__ Q,
                                                                 const T *__restrict__ Kc,
                                                                 const T *__restrict__ Vc, T *__restrict__ A,
                                                                 SelRows sel, int n_q, int n_kv, float scale) {
    constexpr int hd = EPL * 32;
    __shared__ float qs[hd];
    __shared__ float wm[kWarpsA], wl[kWarpsA];
    __shared__ float wacc[kWarpsA][hd];
    griddep_wait();
    griddep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m = blockIdx.x, h = blockIdx.y;
    const int dq = n_q * hd;
    int b, pos;
    sel.locate(m, b, pos);
    T *out = A + (size_t)m * dq + (size_t)h * hd;
    if (pos < 0) {   // not a live row: zeros (the same decision in every thread)
        for (int e = threadIdx.x; e < hd; e += kWarpsA * 32) out[e] = from_f32<T>(0.f);
        return;
    }
    for (int e = threadIdx.x; e < hd; e += kWarpsA * 32) qs[e] = to_f32<T>(Q[(size_t)m * dq + (size_t)h * hd + e]) * scale;
    __syncthreads();
    const int g = h / (n_q / n_kv);
    const size_t kv_stride = (size_t)n_kv * hd;
    const T *kb = Kc + (size_t)b * sel.N * kv_stride + (size_t)g * hd;
    const T *vb = Vc + (size_t)b * sel.N * kv_stride + (size_t)g * hd;
    const int j_begin = (int)((long long)warp * sel.N / kWarpsA), j_end = (int)((long long)(warp + 1) * sel.N / kWarpsA);

    float q[EPL], acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        q[e] = qs[lane * EPL + e];
        acc[e] = 0.f;
    }
    float run_max = -INFINITY, run_sum = 0.f;   // the same in every lane
    int j = j_begin;
    for (; j + 1 < j_end; j += 2) {
        const T *k0 = kb + (size_t)j * kv_stride + lane * EPL, *k1 = k0 + kv_stride;
        const T *v0 = vb + (size_t)j * kv_stride + lane * EPL, *v1 = v0 + kv_stride;
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            s0 = fmaf(q[e], to_f32<T>(k0[e]), s0);
            s1 = fmaf(q[e], to_f32<T>(k1[e]), s1);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            s0 += __shfl_xor_sync(0xffffffffu, s0, o);
            s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        }
        const float nm = fmaxf(run_max, fmaxf(s0, s1));
        const float corr = expf(run_max - nm);
        const float p0 = expf(s0 - nm), p1 = expf(s1 - nm);
        run_sum = run_sum * corr + p0 + p1;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] = fmaf(p1, to_f32<T>(v1[e]), fmaf(p0, to_f32<T>(v0[e]), acc[e] * corr));
        run_max = nm;
    }
    if (j < j_end) {   // odd count: the last key alone
        const T *k0 = kb + (size_t)j * kv_stride + lane * EPL;
        const T *v0 = vb + (size_t)j * kv_stride + lane * EPL;
        float s0 = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) s0 = fmaf(q[e], to_f32<T>(k0[e]), s0);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s0 += __shfl_xor_sync(0xffffffffu, s0, o);
        const float nm = fmaxf(run_max, s0);
        const float corr = expf(run_max - nm);
        const float p0 = expf(s0 - nm);
        run_sum = run_sum * corr + p0;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] = fmaf(p0, to_f32<T>(v0[e]), acc[e] * corr);
        run_max = nm;
    }
    if (lane == 0) {
        wm[warp] = run_max;
        wl[warp] = run_sum;
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) wacc[warp][lane * EPL + e] = acc[e];
    __syncthreads();
    // merge the four warps' (max, sum, accumulator) in warp order
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarpsA; ++w) M = fmaxf(M, wm[w]);
    float den = 0.f, c[kWarpsA];
#pragma unroll
    for (int w = 0; w < kWarpsA; ++w) {
        c[w] = wm[w] == -INFINITY ? 0.f : expf(wm[w] - M);
        den = fmaf(wl[w], c[w], den);
    }
    const float inv = den > 0.f ? 1.0f / den : 0.f;
    for (int e = threadIdx.x; e < hd; e += kWarpsA * 32) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kWarpsA; ++w) v = fmaf(wacc[w][e], c[w], v);
        out[e] = from_f32<T>(v * inv);
    }
}

}  // namespace

template <class T>
cudaError_t attention_simt(const T *Q, const T *Kc, const T *Vc, T *A, SelRows sel, int B, int n_q,
                           int n_kv, int hd, cudaStream_t st) {
    const int M = B * sel.k_max;
    if (M <= 0) return cudaSuccess;
    dim3 grid(M, n_q);
    const float scale = 1.0f / sqrtf((float)hd);
    if (hd == 64)
        return launch_kernel(k_attention_simt<T, 2>, grid, dim3(kWarpsA * 32), 0, st, 1, Q, Kc, Vc, A, sel, n_q,
                             n_kv, scale);
    if (hd == 128)
        return launch_kernel(k_attention_simt<T, 4>, grid, dim3(kWarpsA * 32), 0, st, 1, Q, Kc, Vc, A, sel, n_q,
                             n_kv, scale);
    return cudaErrorInvalidValue;
}

template cudaError_t attention_simt<float>(const float *, const float *, const float *, float *,
                                           SelRows, int, int, int, int, cudaStream_t);
template cudaError_t attention_simt<bf16>(const bf16 *, const bf16 *, const bf16 *, bf16 *, SelRows,
                                          int, int, int, int, cudaStream_t);

}  // namespace dllm
