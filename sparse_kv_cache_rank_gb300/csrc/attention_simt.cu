// attention_simt.cu -- non-causal attention of the selected queries over the whole
// (partially refreshed) cache on the CUDA cores (SPA-Cache, "3. Sparse execution").
// Used for the fp32 configuration.  One warp per (query row, head); each lane holds
// hd/32 dims of q, the score of every key is a warp all-reduce, and the softmax is
// the streaming (running max / running sum) form in fp32.
#include "internal.h"

namespace dllm {
namespace {

template <class T, int EPL>
__global__ void __launch_bounds__(128) k_attention_simt(const T *__restrict__ Q,
                                                        const T *__restrict__ Kc,
                                                        const T *__restrict__ Vc, T *__restrict__ A,
                                                        SelRows sel, int n_q, int n_kv, float scale) {
    constexpr int hd = EPL * 32;
    griddep_wait();
    griddep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y * 4 + warp;
    const int m = blockIdx.x;
    if (h >= n_q) return;
    const int dq = n_q * hd;
    T *out = A + (size_t)m * dq + (size_t)h * hd + lane * EPL;
    int b, pos;
    sel.locate(m, b, pos);
    if (pos < 0) {
#pragma unroll
        for (int e = 0; e < EPL; ++e) out[e] = from_f32<T>(0.f);
        return;
    }
    const int g = h / (n_q / n_kv);
    float q[EPL], acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
        q[e] = to_f32<T>(Q[(size_t)m * dq + (size_t)h * hd + lane * EPL + e]) * scale;
        acc[e] = 0.f;
    }
    float run_max = -INFINITY, run_sum = 0.f;
    const size_t kv_stride = (size_t)n_kv * hd;
    const T *kb = Kc + (size_t)b * sel.N * kv_stride + (size_t)g * hd + lane * EPL;
    const T *vb = Vc + (size_t)b * sel.N * kv_stride + (size_t)g * hd + lane * EPL;
    for (int j = 0; j < sel.N; ++j) {
        float s = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) s = fmaf(q[e], to_f32<T>(kb[(size_t)j * kv_stride + e]), s);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        const float nm = fmaxf(run_max, s);
        const float corr = expf(run_max - nm);
        const float p = expf(s - nm);
        run_sum = run_sum * corr + p;
#pragma unroll
        for (int e = 0; e < EPL; ++e)
            acc[e] = fmaf(p, to_f32<T>(vb[(size_t)j * kv_stride + e]), acc[e] * corr);
        run_max = nm;
    }
    const float inv = 1.0f / run_sum;
#pragma unroll
    for (int e = 0; e < EPL; ++e) out[e] = from_f32<T>(acc[e] * inv);
}

}  // namespace

template <class T>
cudaError_t attention_simt(const T *Q, const T *Kc, const T *Vc, T *A, SelRows sel, int B, int n_q,
                           int n_kv, int hd, cudaStream_t st) {
    const int M = B * sel.k_max;
    if (M <= 0) return cudaSuccess;
    dim3 grid(M, (n_q + 3) / 4);
    const float scale = 1.0f / sqrtf((float)hd);
    if (hd == 64)
        launch_kernel(k_attention_simt<T, 2>, grid, dim3(128), 0, st, 1, Q, Kc, Vc, A, sel, n_q, n_kv, scale);
    else if (hd == 128)
        launch_kernel(k_attention_simt<T, 4>, grid, dim3(128), 0, st, 1, Q, Kc, Vc, A, sel, n_q, n_kv, scale);
    else
        return cudaErrorInvalidValue;
    return cudaGetLastError();
}

template cudaError_t attention_simt<float>(const float *, const float *, const float *, float *,
                                           SelRows, int, int, int, int, cudaStream_t);
template cudaError_t attention_simt<bf16>(const bf16 *, const bf16 *, const bf16 *, bf16 *, SelRows,
                                          int, int, int, int, cudaStream_t);

}  // namespace dllm
