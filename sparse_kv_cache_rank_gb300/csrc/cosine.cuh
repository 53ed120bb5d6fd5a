// cosine.cuh -- the cosine drift of one proxy row by one warp (SPA-Cache, "1. Update
// identification via singular proxy"), shared by the cosine kernel and the layer step's
// fused drift + selection kernel, so that both give bit-identical drifts.
//
// drift = 1 - cos(cur, cached), evaluated as |cur/|cur| - cached/|cached||^2 / 2, which
// equals 1 - cos for unit vectors and keeps the small drifts of nearly unchanged rows
// free of the cancellation in 1 - dot/norm.  Identical inputs give exactly 0; both norms
// zero -> 0, one zero -> 1; clamped to [0, 2].  With nparts > 1 the proxy is first summed
// from the K-slice partials in slice order (the same order every call, so identical
// inputs still give identical proxies) and stored to cur.
#pragma once

#include "internal.h"

namespace dllm {

// Row `row` of rows x r (r % 32 == 0, r <= 128 * MAXCH): float4 chunk lane + 32u of the
// row in lane's registers for both passes.  Returns the drift in every lane.
template <int MAXCH>
__device__ __forceinline__ float cosine_row(const float *__restrict__ parts, int nparts,
                                            const float *__restrict__ cached, float *__restrict__ cur,
                                            long row, long rows, int r, int lane) {
    const int nch = r >> 2;
    const size_t stride4 = (size_t)rows * nch;
    const float4 *p4 = reinterpret_cast<const float4 *>(parts) + (size_t)row * nch;
    float4 *a4 = reinterpret_cast<float4 *>(cur + row * r);
    const float4 *c4 = reinterpret_cast<const float4 *>(cached + row * r);
    float4 xs[MAXCH], cs[MAXCH];
    float na = 0.f, nc = 0.f;
    // for each chunk every partial load is issued before the first add; adds in slice order
#pragma unroll
    for (int u = 0; u < MAXCH; ++u) {
        const int ch = lane + 32 * u;
        if (ch >= nch) break;
        float4 x;
        const float4 cc = __ldcg(c4 + ch);
        if (nparts > 1) {
            float4 t[8];
#pragma unroll
            for (int z = 0; z < 8; ++z)
                if (z < nparts) t[z] = __ldcg(p4 + (size_t)z * stride4 + ch);
            x = t[0];
#pragma unroll
            for (int z = 1; z < 8; ++z)
                if (z < nparts) {
                    x.x += t[z].x;
                    x.y += t[z].y;
                    x.z += t[z].z;
                    x.w += t[z].w;
                }
            for (int z = 8; z < nparts; ++z) {
                const float4 y = __ldcg(p4 + (size_t)z * stride4 + ch);
                x.x += y.x;
                x.y += y.y;
                x.z += y.z;
                x.w += y.w;
            }
            a4[ch] = x;
        } else {
            x = __ldcg(a4 + ch);
        }
        xs[u] = x;
        cs[u] = cc;
        na = fmaf(x.x, x.x, fmaf(x.y, x.y, fmaf(x.z, x.z, fmaf(x.w, x.w, na))));
        nc = fmaf(cc.x, cc.x, fmaf(cc.y, cc.y, fmaf(cc.z, cc.z, fmaf(cc.w, cc.w, nc))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        na += __shfl_xor_sync(0xffffffffu, na, o);
        nc += __shfl_xor_sync(0xffffffffu, nc, o);
    }
    if (na == 0.f && nc == 0.f) return 0.f;
    if (na == 0.f || nc == 0.f) return 1.f;
    const float ia = 1.0f / sqrtf(na), ic = 1.0f / sqrtf(nc);
    float s = 0.f;
#pragma unroll
    for (int u = 0; u < MAXCH; ++u) {   // the chunks this lane summed above
        if (lane + 32 * u >= nch) break;
        const float4 x = xs[u], cc = cs[u];
        // separately rounded products (no FMA contraction): equal inputs give t == 0
        const float t0 = __fsub_rn(__fmul_rn(x.x, ia), __fmul_rn(cc.x, ic));
        const float t1 = __fsub_rn(__fmul_rn(x.y, ia), __fmul_rn(cc.y, ic));
        const float t2 = __fsub_rn(__fmul_rn(x.z, ia), __fmul_rn(cc.z, ic));
        const float t3 = __fsub_rn(__fmul_rn(x.w, ia), __fmul_rn(cc.w, ic));
        s = fmaf(t0, t0, fmaf(t1, t1, fmaf(t2, t2, fmaf(t3, t3, s))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    return fminf(fmaxf(0.5f * s, 0.f), 2.f);
}

}  // namespace dllm
