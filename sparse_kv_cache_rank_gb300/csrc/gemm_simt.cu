// gemm_simt.cu -- fp32 GEMM on the CUDA cores for the fp32 configuration
// (tensor-core TF32 would not meet fp32 accuracy).  Same contract and epilogues
// as the tensor-core GEMM: acc[f, m] = <W[f, :], X[m, :]>.
//
// Tile: 64 weight rows x 64 tokens, K step 16.  Thread (warp w, lane l) owns
// weight rows l and l + 32 and tokens 8w .. 8w + 7, so at the epilogue each warp
// holds 32 consecutive weight rows of one token, as the epilogues expect.
#include "internal.h"

namespace dllm {
namespace {

constexpr int TF = 64, TM = 64, TK = 16;

template <class Epi>
__global__ void __launch_bounds__(256) k_gemm_simt(const float *__restrict__ W, int N_out, int K,
                                                   const float *__restrict__ X, int M_tok, const Epi epi) {
    __shared__ float Ws[TK][TF + 1];
    __shared__ float Xs[TK][TM + 1];
    griddep_wait();
    griddep_launch();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * TM, f0 = blockIdx.y * TF;
    float acc[2][8];
#pragma unroll
    for (int g = 0; g < 2; ++g)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[g][j] = 0.f;

    for (int k0 = 0; k0 < K; k0 += TK) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int id = threadIdx.x + i * 256;
            const int r = id / TK, k = id % TK;
            const int gk = k0 + k;
            const int gf = f0 + r, gm = m0 + r;
            Ws[k][r] = (gf < N_out && gk < K) ? W[(size_t)gf * K + gk] : 0.f;
            Xs[k][r] = (gm < M_tok && gk < K) ? X[(size_t)gm * K + gk] : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < TK; ++k) {
            const float a0 = Ws[k][lane], a1 = Ws[k][lane + 32];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float x = Xs[k][warp * 8 + j];
                acc[0][j] = fmaf(a0, x, acc[0][j]);
                acc[1][j] = fmaf(a1, x, acc[1][j]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int m = m0 + warp * 8 + j;
        if (m >= M_tok) break;
        int b = 0, pos = -1;
        if (Epi::kSel) epi.sel.locate(m, b, pos);
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            if (f0 + g * 32 < N_out) {
                const typename Epi::Feat F = epi.feat(f0 + g * 32 + lane);
                epi(F, m, b, pos, acc[g][j], epi.pre(F, m, b, pos));
            }
        }
    }
}

}  // namespace

template <class Epi>
cudaError_t gemm_simt(const float *W, int N_out, int K, const float *X, int M_tok, const Epi &epi,
                      cudaStream_t st) {
    if (M_tok <= 0 || N_out <= 0) return cudaSuccess;
    if (N_out % 32 != 0) return cudaErrorInvalidValue;
    dim3 grid((M_tok + TM - 1) / TM, (N_out + TF - 1) / TF);
    return launch_kernel(k_gemm_simt<Epi>, grid, dim3(256), 0, st, 1, W, N_out, K, X, M_tok, epi);
}

template cudaError_t gemm_simt<EpiStoreF32>(const float *, int, int, const float *, int,
                                            const EpiStoreF32 &, cudaStream_t);
template cudaError_t gemm_simt<EpiQKV<float>>(const float *, int, int, const float *, int,
                                              const EpiQKV<float> &, cudaStream_t);
template cudaError_t gemm_simt<EpiResidual<float>>(const float *, int, int, const float *, int,
                                                   const EpiResidual<float> &, cudaStream_t);
template cudaError_t gemm_simt<EpiSwiGLU<float>>(const float *, int, int, const float *, int,
                                                 const EpiSwiGLU<float> &, cudaStream_t);
template cudaError_t gemm_simt<EpiDownScatter<float>>(const float *, int, int, const float *, int,
                                                      const EpiDownScatter<float> &, cudaStream_t);

}  // namespace dllm
