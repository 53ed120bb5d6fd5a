// rownorm.cuh -- block-level RMSNorm of one row (256 threads) and the vector helpers it
// uses, shared by the row kernels (gather + norm of the selected rows, second norm, final
// norm) and the fused selection + gather kernel.
#pragma once

#include "internal.h"

namespace dllm {
namespace rownorm {

template <int NT>
__device__ __forceinline__ float block_sum(float v, float *red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.f;
    if (threadIdx.x < 32) {
        t = threadIdx.x < NT / 32 ? red[threadIdx.x] : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (threadIdx.x == 0) red[32] = t;
    }
    __syncthreads();
    return red[32];
}

// 16-byte vectors of a row: 8 bf16 or 4 fp32 values.
template <class T> struct Vec16;
template <> struct Vec16<bf16> {
    static constexpr int n = 8;
    __device__ static void unpack(const uint4 &u, float *x) {
        const __nv_bfloat162 *p = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __bfloat1622float2(p[i]);
            x[2 * i] = f.x;
            x[2 * i + 1] = f.y;
        }
    }
};
template <> struct Vec16<float> {
    static constexpr int n = 4;
    __device__ static void unpack(const uint4 &u, float *x) {
        x[0] = __uint_as_float(u.x);
        x[1] = __uint_as_float(u.y);
        x[2] = __uint_as_float(u.z);
        x[3] = __uint_as_float(u.w);
    }
};

template <int Bytes> struct VecBytes;
template <> struct VecBytes<8> { using type = uint2; };
template <> struct VecBytes<16> { using type = uint4; };

// out = RMSNorm(row) * gamma for one row of d values, 256 threads.  Rows whose 16-byte
// vectors fit 4 per thread are read once into registers with 16-byte loads (row, gamma
// and out 16-byte aligned); others take the plain loop.
template <class TI, class TO>
__device__ __forceinline__ void norm_row(const TI *__restrict__ row, int d, const TO *__restrict__ gamma,
                                         float eps, TO *__restrict__ out, float *red) {
    constexpr int V = Vec16<TI>::n, kVPT = 4;
    const int nv = d / V;
    if (d % V == 0 && d % Vec16<TO>::n == 0 && nv <= 256 * kVPT) {
        uint4 xv[kVPT];
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < kVPT; ++j) {
            const int vi = threadIdx.x + j * 256;
            if (vi < nv) {
                xv[j] = reinterpret_cast<const uint4 *>(row)[vi];
                float x[V];
                Vec16<TI>::unpack(xv[j], x);
#pragma unroll
                for (int i = 0; i < V; ++i) ss = fmaf(x[i], x[i], ss);
            }
        }
        ss = block_sum<256>(ss, red);
        const float inv = 1.0f / sqrtf(ss / (float)d + eps);
#pragma unroll
        for (int j = 0; j < kVPT; ++j) {
            const int vi = threadIdx.x + j * 256;
            if (vi < nv) {
                float x[V];
                Vec16<TI>::unpack(xv[j], x);
                using Chunk = typename VecBytes<V * sizeof(TO)>::type;   // V outputs / gammas
                Chunk gc = *reinterpret_cast<const Chunk *>(gamma + (size_t)vi * V);
                const TO *gv = reinterpret_cast<const TO *>(&gc);
                Chunk oc;
                TO *ov = reinterpret_cast<TO *>(&oc);
#pragma unroll
                for (int i = 0; i < V; ++i) ov[i] = from_f32<TO>(x[i] * inv * to_f32<TO>(gv[i]));
                *reinterpret_cast<Chunk *>(out + (size_t)vi * V) = oc;
            }
        }
        return;
    }
    float ss = 0.f;
    for (int e = threadIdx.x; e < d; e += 256) {
        const float x = to_f32<TI>(row[e]);
        ss = fmaf(x, x, ss);
    }
    ss = block_sum<256>(ss, red);
    const float inv = 1.0f / sqrtf(ss / (float)d + eps);
    for (int e = threadIdx.x; e < d; e += 256)
        out[e] = from_f32<TO>(to_f32<TI>(row[e]) * inv * to_f32<TO>(gamma[e]));
}

}  // namespace rownorm
}  // namespace dllm
