// gemm_simt.cu -- fp32 GEMM on the CUDA cores for the fp32 configuration
// (tensor-core TF32 would not meet fp32 accuracy).  Same contract and epilogues
// as the tensor-core GEMM: acc[f, m] = <W[f, :], X[m, :]>.
//
// Tile: 32 weight rows x 32 tokens, K step 32; the next step's tile is loaded into
// registers while the current one is multiplied.  Thread (warp w, lane l) owns weight
// row l and tokens 4w .. 4w + 3, so at the epilogue each warp holds 32 consecutive
// weight rows of one token, as the epilogues expect.  The small layers this path serves
// have few tiles, so when the tiles alone leave most SMs idle the K range is split over
// a thread-block cluster (up to 8 CTAs): the CTAs sum their partial tiles through
// distributed shared memory in rank order (a fixed order) and each finishes a share of
// the tile's tokens.
#include "internal.h"

namespace dllm {
namespace {

constexpr int TF = 32, TM = 32, TK = 32;
constexpr int kT = 256;

template <class Epi>
__global__ void __launch_bounds__(kT) k_gemm_simt(const float *__restrict__ W, int N_out, int K,
                                                  const float *__restrict__ X, int M_tok, const Epi epi,
                                                  int splits, unsigned *zero, int nzero) {
    // rows padded to 36 words: 16-byte aligned for the float4 reads of Xs, and the
    // transposed stores below (rows lk + 8i, columns lr) still hit 32 distinct banks
    __shared__ __align__(16) float Ws[TK][TF + 4];
    __shared__ __align__(16) float Xs[TK][TM + 4];
    __shared__ float part[TM][TF];   // this CTA's partial tile (K split)
    griddep_wait();
    griddep_launch();
    // counters of the kernel that follows, cleared once the previous kernel is done
    if (zero && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
        for (int i = threadIdx.x; i < nzero; i += kT) zero[i] = 0u;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * TM, f0 = blockIdx.y * TF;
    const int split = splits > 1 ? (int)cluster_ctarank() : 0;
    const int nkt = (K + TK - 1) / TK;
    const int kt0 = (int)((long long)split * nkt / splits), kt1 = (int)((long long)(split + 1) * nkt / splits);

    // loads: row lr of the W and X tiles, K offsets lk + 8 i (eight threads per 32-byte
    // row segment)
    const int lr = threadIdx.x >> 3, lk = threadIdx.x & 7;
    const bool w_row = f0 + lr < N_out, x_row = m0 + lr < M_tok;
    const float *wp = W + (size_t)(f0 + lr) * K;
    const float *xp = X + (size_t)(m0 + lr) * K;
    float rw[4], rx[4];
    auto load = [&](int kt) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int k = kt * TK + lk + 8 * i;
            rw[i] = (w_row && k < K) ? wp[k] : 0.f;
            rx[i] = (x_row && k < K) ? xp[k] : 0.f;
        }
    };
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (kt0 < kt1) load(kt0);
    for (int kt = kt0; kt < kt1; ++kt) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            Ws[lk + 8 * i][lr] = rw[i];
            Xs[lk + 8 * i][lr] = rx[i];
        }
        __syncthreads();
        if (kt + 1 < kt1) load(kt + 1);   // in flight while this tile is multiplied
#pragma unroll
        for (int k = 0; k < TK; ++k) {
            const float a = Ws[k][lane];
            const float4 x = *reinterpret_cast<const float4 *>(&Xs[k][warp * 4]);   // broadcast
            acc[0] = fmaf(a, x.x, acc[0]);
            acc[1] = fmaf(a, x.y, acc[1]);
            acc[2] = fmaf(a, x.z, acc[2]);
            acc[3] = fmaf(a, x.w, acc[3]);
        }
        __syncthreads();
    }

    // f0 + lane < N_out always (N_out % 32 == 0); warp-uniform conditions only below, the
    // epilogues shuffle between neighbouring lanes
    const typename Epi::Feat F = epi.feat(f0 + lane);
    if (splits == 1) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int m = m0 + warp * 4 + j;
            if (m >= M_tok) break;
            int b = 0, pos = -1;
            if (Epi::kSel) epi.sel.locate(m, b, pos);
            epi(F, m, b, pos, acc[j], epi.pre(F, m, b, pos));
        }
        return;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) part[warp * 4 + j][lane] = acc[j];
    cluster_sync_all();
    // rank `split` finishes tokens [t0, t1) of the tile: the sum of every rank's partial
    const int t0 = split * TM / splits, t1 = (split + 1) * TM / splits;
    for (int t = t0 + warp; t < t1; t += kT / 32) {
        const uint32_t local = smem_u32(&part[t][lane]);
        float v = 0.f;
        for (int q = 0; q < splits; ++q) v += ld_dsmem_f32(mapa_shared(local, (uint32_t)q));
        const int m = m0 + t;
        if (m < M_tok) {
            int b = 0, pos = -1;
            if (Epi::kSel) epi.sel.locate(m, b, pos);
            epi(F, m, b, pos, v, epi.pre(F, m, b, pos));
        }
    }
    cluster_sync_all();   // peers may still read this CTA's partial tile
}

}  // namespace

template <class Epi>
cudaError_t gemm_simt(const float *W, int N_out, int K, const float *X, int M_tok, const Epi &epi,
                      cudaStream_t st, unsigned *zero, int nzero) {
    if (M_tok <= 0 || N_out <= 0) return cudaSuccess;
    if (N_out % 32 != 0 || K <= 0) return cudaErrorInvalidValue;
    const dim3 tiles((M_tok + TM - 1) / TM, N_out / TF);
    const long long n_tiles = (long long)tiles.x * tiles.y;
    const int sms = num_sms();
    const int nkt = (K + TK - 1) / TK;
    // K split (cluster of s CTAs) when the tiles fill fewer than the SMs: about two CTAs
    // per SM, at least two K steps per CTA
    int s = n_tiles >= sms ? 1 : (int)(2LL * sms / n_tiles);
    s = s < 1 ? 1 : (s > 8 ? 8 : s);
    while (s > 1 && nkt / s < 2) --s;
    return launch_kernel(k_gemm_simt<Epi>, dim3(tiles.x, tiles.y, s), dim3(kT), 0, st, s, W, N_out, K, X, M_tok,
                         epi, s, zero, zero ? nzero : 0);
}

template cudaError_t gemm_simt<EpiStoreF32>(const float *, int, int, const float *, int,
                                            const EpiStoreF32 &, cudaStream_t, unsigned *, int);
template cudaError_t gemm_simt<EpiQKV<float>>(const float *, int, int, const float *, int,
                                              const EpiQKV<float> &, cudaStream_t, unsigned *, int);
template cudaError_t gemm_simt<EpiResidual<float>>(const float *, int, int, const float *, int,
                                                   const EpiResidual<float> &, cudaStream_t, unsigned *, int);
template cudaError_t gemm_simt<EpiSwiGLU<float>>(const float *, int, int, const float *, int,
                                                 const EpiSwiGLU<float> &, cudaStream_t, unsigned *, int);
template cudaError_t gemm_simt<EpiDownScatter<float>>(const float *, int, int, const float *, int,
                                                      const EpiDownScatter<float> &, cudaStream_t, unsigned *, int);

}  // namespace dllm
