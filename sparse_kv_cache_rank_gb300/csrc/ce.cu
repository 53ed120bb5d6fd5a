// ce.cu -- confidence extrapolation ("Efficient diffusion LLMs via temporal-spatial parallel
// decoding and confidence extrapolation", 2. Confidence Extrapolation): every token's top-1
// confidence is the noisy observation of a latent (level, velocity) state, tracked by a
// constant-velocity Kalman filter; the forecast h steps ahead has mean l + h v and variance
// P00 + 2h P01 + h^2 P11; an undecided token is committed early when the z-lower bound of
// some forecast within its horizon reaches c_min, the horizon being min(h_max, committed
// positions to its left in the block).  One CTA per sequence, one thread per block position;
// the left-context counts come from a block-wide exclusive scan.
#include <math.h>

#include "internal.h"

namespace dllm {
namespace {

__global__ void __launch_bounds__(1024)
    k_ce_step(const float *__restrict__ conf, const uint8_t *__restrict__ seen,
              const uint8_t *__restrict__ undecided, const uint8_t *__restrict__ committed,
              float *__restrict__ state, uint8_t *__restrict__ early, int M, CEParams p) {
    __shared__ int wsum[32];
    griddep_wait();
    griddep_launch();
    const int b = blockIdx.x, i = threadIdx.x;
    const int lane = i & 31, warp = i >> 5;
    const size_t t = (size_t)b * M + i;

    // committed positions left of i (exclusive scan over the block)
    const int cm = i < M && committed[t] != 0;
    int incl = cm;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int nw = (blockDim.x + 31) >> 5;
        const int w = lane < nw ? wsum[lane] : 0;
        int s = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        wsum[lane] = s - w;
    }
    __syncthreads();
    if (i >= M) return;
    const int cover = wsum[warp] + incl - cm;

    float *st = state + t * 5;
    const float c = conf[t];
    float l, v, p00, p01, p11;
    if (seen[t]) {
        l = st[0];
        v = st[1];
        p00 = st[2];
        p01 = st[3];
        p11 = st[4];
        // predict: x- = F x, P- = F P F^T + diag(q_l, q_v), F = [[1, 1], [0, 1]]
        const float lm = l + v;
        const float m00 = p00 + 2.f * p01 + p11 + p.q_l;
        const float m01 = p01 + p11;
        const float m11 = p11 + p.q_v;
        // update with the observed level
        const float S = m00 + p.R;
        const float k0 = m00 / S, k1 = m01 / S;
        const float e = c - lm;
        l = lm + k0 * e;
        v = v + k1 * e;
        p00 = (1.f - k0) * m00;
        p01 = (1.f - k0) * m01;
        p11 = m11 - k1 * m01;
    } else {   // first observation of this token
        l = c;
        v = 0.f;
        p00 = p.R;
        p01 = 0.f;
        p11 = p.p_v0;
    }
    st[0] = l;
    st[1] = v;
    st[2] = p00;
    st[3] = p01;
    st[4] = p11;

    uint8_t go = 0;
    if (undecided[t]) {
        const int H = cover < p.h_max ? cover : p.h_max;
        for (int h = 1; h <= H; ++h) {
            const float fh = (float)h;
            const float mean = l + fh * v;
            const float var = p00 + 2.f * fh * p01 + fh * fh * p11;
            if (mean - p.z * sqrtf(fmaxf(var, 0.f)) >= p.c_min) go = 1;
        }
    }
    early[t] = go;
}

}  // namespace

cudaError_t ce_step(const float *conf, const uint8_t *seen, const uint8_t *undecided,
                    const uint8_t *committed, float *state, uint8_t *early, int B, int M,
                    const CEParams &p, cudaStream_t st) {
    if (B <= 0 || M <= 0) return cudaSuccess;
    if (M > 1024) return cudaErrorInvalidValue;
    const int threads = (M + 31) / 32 * 32;
    return launch_kernel(k_ce_step, dim3((unsigned)B), dim3((unsigned)threads), 0, st, 1, conf, seen,
                         undecided, committed, state, early, M, p);
}

}  // namespace dllm
