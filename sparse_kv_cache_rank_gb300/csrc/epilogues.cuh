// epilogues.cuh -- output stages of the refresh GEMMs (SPA-Cache, "3. Sparse execution").
//
// A GEMM computes acc[f, m] = <W[f, :], X[m, :]> for weight row f and token row m
// and hands every accumulator to an epilogue.  Both GEMM kernels call the epilogue
// with a FULL warp whose 32 lanes hold 32 consecutive weight rows (f = f0 + lane,
// f0 % 32 == 0) of the same token m, so that neighbouring rows (f, f ^ 1) can be
// combined with one shuffle:
//   * rotary pairs (dims i and i + hd/2 of a head) are packed as rows 2i, 2i+1;
//   * SwiGLU gate j and up j are packed as rows 2j, 2j+1.
// Token rows are the flattened selection m = b * k_max + s; a row is live when
// s < min(count[b], k_max) and then refers to sequence position pos = idx[b, s].
//
// Interface of an epilogue E:
//   E::kSel            the GEMM resolves (b, pos) of every token column (else b = 0, pos = -1)
//   E::Feat feat(f)    per-weight-row constants, computed once per thread
//   float2 pre(F, m, b, pos)            the global values one output needs (residual
//                                       input, rotary cos/sin); the GEMM issues them for a
//                                       batch of columns before consuming any
//   operator()(F, m, b, pos, acc, pre)  writes the output(s)
#pragma once

#include "common.cuh"

namespace dllm {

struct SelRows {
    const int32_t *idx;     // [B, N]
    const int32_t *count;   // [B]
    int k_max, N;

    // Sequence b and cache position of flattened row m; pos < 0 when not live.
    __device__ __forceinline__ void locate(int m, int &b, int &pos) const {
        b = m / k_max;
        const int s = m - b * k_max;
        int c = count[b];
        c = c < k_max ? c : k_max;
        pos = -1;
        if (s < c) {
            const int p = idx[(size_t)b * N + s];
            pos = (p >= 0 && p < N) ? p : -1;
        }
    }
};

struct FeatRow {
    int f;
};

// out[m, f] = acc (fp32), for f < n_valid.  Singular proxy and plain GEMM.
struct EpiStoreF32 {
    static constexpr bool kSel = false;
    static constexpr bool kTileReduce = false;
    static constexpr bool kColScale = false;
    using Feat = FeatRow;
    SelRows sel;
    float *out;
    int ld, n_valid;
    __device__ __forceinline__ Feat feat(int f) const { return {f}; }
    __device__ __forceinline__ float2 pre(const Feat &, int, int, int) const { return {0.f, 0.f}; }
    __device__ __forceinline__ void operator()(const Feat &F, int m, int, int, float acc, float2) const {
        if (F.f < n_valid) out[(size_t)m * ld + F.f] = acc;
    }
};

// Singular proxy with its cosine drift (SPA-Cache, "1. Update identification via singular
// proxy"): cur[m, :] = acc over the proxy's r <= 128 features (one weight tile) and
// drift[m] = 1 - cos(cur[m], cached[m]), computed as 0.5 |cur/|cur| - cached/|cached||^2
// (exactly 0 for identical proxies), 0 when both are zero, 1 when exactly one is, clamped
// to [0, 2].  The drift needs every feature of a token, so the GEMM runs it only without a
// K split (each CTA's accumulators hold a token's whole proxy): it hands the epilogue whole
// 16-column chunks (kCosine) and reduces over the 128 TMEM lanes itself, and the operator
// below is never called.
struct EpiCosine {
    static constexpr bool kSel = false;
    static constexpr bool kTileReduce = false;
    static constexpr bool kColScale = false;
    static constexpr bool kCosine = true;
    using Feat = FeatRow;
    SelRows sel;
    float *cur;            // [rows, r]
    const float *cached;   // [rows, r]
    float *drift;          // [rows]
    int r;
    __device__ __forceinline__ Feat feat(int f) const { return {f}; }
    __device__ __forceinline__ float2 pre(const Feat &, int, int, int) const { return {0.f, 0.f}; }
    __device__ __forceinline__ void operator()(const Feat &, int, int, int, float, float2) const {}
};

// [Q | K | V] rows -> rotary embedding at the token's position; Q to the compact
// query buffer, K and V scattered into the cache rows.  rope_cs [M, hd/2] holds
// (cos, sin) of pos * theta^(-2i/hd) for every selected row (written by the gather).
template <class T>
struct EpiQKV {
    static constexpr bool kSel = true;
    static constexpr bool kTileReduce = false;
    static constexpr bool kColScale = false;
    SelRows sel;
    T *Q;               // [M, n_q*hd]
    T *Kc, *Vc;         // [B, N, n_kv, hd]
    const float2 *rope_cs;
    int n_q, n_kv, hd, use_rope;

    struct Feat {
        int region;     // 0 Q, 1 K, 2 V
        int col;        // head * hd + dim: output column inside Q / K / V
        int i;          // rotary pair index
        int odd;        // second half of the pair
    };
    __device__ __forceinline__ Feat feat(int f) const {
        const int dq = n_q * hd, dkv = n_kv * hd;
        Feat F;
        int g;
        if (f < dq) { F.region = 0; g = f; }
        else if (f < dq + dkv) { F.region = 1; g = f - dq; }
        else { F.region = 2; g = f - dq - dkv; }
        const int head = g / hd, p = g - head * hd;
        F.i = p >> 1;
        F.odd = p & 1;
        F.col = head * hd + (F.odd ? F.i + (hd >> 1) : F.i);
        return F;
    }
    __device__ __forceinline__ float2 pre(const Feat &F, int m, int, int) const {
        if (!use_rope || F.region == 2) return {1.f, 0.f};
        return rope_cs[(size_t)m * (hd >> 1) + F.i];
    }
    __device__ __forceinline__ void operator()(const Feat &F, int m, int b, int pos, float acc,
                                               float2 cs) const {
        const float partner = __shfl_xor_sync(0xffffffffu, acc, 1);
        const float out = F.odd ? fmaf(acc, cs.x, partner * cs.y) : fmaf(acc, cs.x, -partner * cs.y);
        if (F.region == 0) {
            Q[(size_t)m * (n_q * hd) + F.col] = from_f32<T>(out);
        } else if (pos >= 0) {
            T *dst = F.region == 1 ? Kc : Vc;
            dst[((size_t)b * sel.N + pos) * (size_t)(n_kv * hd) + F.col] = from_f32<T>(out);
        }
    }
};

// h1[m, f] = H_in[b, pos, f] + acc (fp32); 0 for rows that are not live.
template <class T>
struct EpiResidual {
    static constexpr bool kSel = true;
    static constexpr bool kTileReduce = false;
    static constexpr bool kColScale = false;
    using Feat = FeatRow;
    SelRows sel;
    float *h1;          // [M, d]
    const T *H_in;      // [B, N, d]
    int d;
    __device__ __forceinline__ Feat feat(int f) const { return {f}; }
    __device__ __forceinline__ float2 pre(const Feat &F, int, int b, int pos) const {
        return {pos >= 0 ? to_f32<T>(H_in[((size_t)b * sel.N + pos) * d + F.f]) : 0.f, 0.f};
    }
    __device__ __forceinline__ void operator()(const Feat &F, int m, int, int pos, float acc,
                                               float2 hin) const {
        h1[(size_t)m * d + F.f] = pos >= 0 ? hin.x + acc : 0.f;
    }
};

// The O projection with the second RMSNorm folded in: h1[m, f] = H_in[b, pos, f] + acc
// (fp32, the down projection's residual), Xh[m, f] = bf16(h1 * gamma2[f]) (the gate/up
// GEMM's operand: RMSNorm's per-row scale is applied to its accumulators instead), and
// ss[f / 32][m] = sum of h1^2 over the warp's 32 features (fixed-order partial sums of the
// row's squares, summed in order by EpiSwiGLUNorm).  0 for rows that are not live.
template <class T>
struct EpiResidualNorm {
    static constexpr bool kSel = true;
    static constexpr bool kTileReduce = false;
    static constexpr bool kColScale = false;
    struct Feat {
        int f;
        float g;
    };
    SelRows sel;
    float *h1;          // [M, d]
    T *Xh;              // [M, d]
    float *ss;          // [d / 32][M]
    const T *H_in;      // [B, N, d]
    const T *gamma2;    // [d]
    int d, M;
    __device__ __forceinline__ Feat feat(int f) const { return {f, to_f32<T>(gamma2[f])}; }
    __device__ __forceinline__ float2 pre(const Feat &F, int, int b, int pos) const {
        return {pos >= 0 ? to_f32<T>(H_in[((size_t)b * sel.N + pos) * d + F.f]) : 0.f, 0.f};
    }
    __device__ __forceinline__ void operator()(const Feat &F, int m, int, int pos, float acc,
                                               float2 hin) const {
        const float v = pos >= 0 ? hin.x + acc : 0.f;
        h1[(size_t)m * d + F.f] = v;
        Xh[(size_t)m * d + F.f] = from_f32<T>(v * F.g);
        float sq = v * v;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
        if ((F.f & 31) == 0) ss[(size_t)(F.f >> 5) * M + m] = sq;
    }
};

// Rows 2j (gate) and 2j+1 (up): U[m, j] = SiLU(gate) * up.
template <class T>
struct EpiSwiGLU {
    static constexpr bool kSel = false;
    static constexpr bool kTileReduce = false;
    static constexpr bool kColScale = false;
    using Feat = FeatRow;
    SelRows sel;
    T *U;               // [M, F]
    int F;
    __device__ __forceinline__ Feat feat(int f) const { return {f}; }
    __device__ __forceinline__ float2 pre(const Feat &, int, int, int) const { return {0.f, 0.f}; }
    __device__ __forceinline__ void operator()(const Feat &Fr, int m, int, int, float acc, float2) const {
        const float partner = __shfl_xor_sync(0xffffffffu, acc, 1);
        if ((Fr.f & 1) == 0) U[(size_t)m * F + (Fr.f >> 1)] = from_f32<T>(silu(acc) * partner);
    }
};

// SwiGLU on the RMSNorm'd rows when the operand is bf16(h1 * gamma2) (EpiResidualNorm):
// every accumulator of token m is first scaled by 1 / sqrt(mean(h1[m]^2) + eps), from the
// fixed-order sum of the row's partial squares.  The GEMM evaluates col_scale(m) once per
// token column and passes it in the column's position slot (this epilogue selects nothing).
template <class T>
struct EpiSwiGLUNorm {
    static constexpr bool kSel = false;
    static constexpr bool kTileReduce = false;
    static constexpr bool kColScale = true;
    using Feat = FeatRow;
    SelRows sel;
    T *U;               // [M, F]
    const float *ss;    // [d / 32][M]
    int F, d, M;
    float eps;
    __device__ __forceinline__ float col_scale(int m) const {
        float s = 0.f;
        for (int p = 0; p < d / 32; ++p) s += ss[(size_t)p * M + m];
        return 1.0f / sqrtf(s / (float)d + eps);
    }
    __device__ __forceinline__ Feat feat(int f) const { return {f}; }
    __device__ __forceinline__ float2 pre(const Feat &, int, int, int) const { return {0.f, 0.f}; }
    __device__ __forceinline__ void operator()(const Feat &Fr, int m, int, int scale_bits, float acc, float2) const {
        const float x = acc * __int_as_float(scale_bits);
        const float partner = __shfl_xor_sync(0xffffffffu, x, 1);
        if ((Fr.f & 1) == 0) U[(size_t)m * F + (Fr.f >> 1)] = from_f32<T>(silu(x) * partner);
    }
};

// H_out_cache[b, pos, f] = h1[m, f] + acc for live rows.
template <class T>
struct EpiDownScatter {
    static constexpr bool kSel = true;
    static constexpr bool kTileReduce = false;
    static constexpr bool kColScale = false;
    using Feat = FeatRow;
    SelRows sel;
    T *H_out;           // [B, N, d]
    const float *h1;    // [M, d]
    int d;
    __device__ __forceinline__ Feat feat(int f) const { return {f}; }
    __device__ __forceinline__ float2 pre(const Feat &F, int m, int, int pos) const {
        return {pos >= 0 ? h1[(size_t)m * d + F.f] : 0.f, 0.f};
    }
    __device__ __forceinline__ void operator()(const Feat &F, int, int b, int pos, float acc,
                                               float2 h) const {
        if (pos >= 0) H_out[((size_t)b * sel.N + pos) * d + F.f] = from_f32<T>(h.x + acc);
    }
};

// Online softmax state of a set of logits l_i (EntropyCache, "How EntropyCache works",
// step 2; TSPD "Input features"): m = max, a = its lowest index, s = sum e^(l - m),
// t = sum (l - m) e^(l - m); then p_max = 1/s and entropy = ln s - t/s.  States of
// disjoint sets merge exactly under a change of reference maximum.  s == 0: empty set.
struct VocabState {
    float m, s, t;
    int a;
};

__device__ __forceinline__ VocabState vocab_merge(VocabState x, VocabState y) {
    if (y.s == 0.f) return x;
    if (x.s == 0.f) return y;
    if (y.m > x.m || (y.m == x.m && y.a < x.a)) {
        const VocabState tmp = x;
        x = y;
        y = tmp;
    }
    // x holds the larger maximum (lower index on equal maxima)
    const float c = expf(y.m - x.m);
    VocabState r;
    r.m = x.m;
    r.a = x.a;
    r.s = x.s + y.s * c;
    r.t = x.t + c * (y.t + (y.m - x.m) * y.s);
    return r;
}

// LM head fused with the vocabulary statistics: instead of storing logits, the GEMM
// reduces each weight tile (128 vocabulary rows) to one VocabState per token row:
// part[m * tiles + tile].  Rows at or past V are not part of any state.
struct EpiVocabStats {
    static constexpr bool kSel = false;
    static constexpr bool kTileReduce = true;
    static constexpr bool kColScale = false;
    using Feat = FeatRow;
    SelRows sel;
    VocabState *part;   // [M_tok][tiles]
    int tiles;
    __device__ __forceinline__ Feat feat(int f) const { return {f}; }
    __device__ __forceinline__ float2 pre(const Feat &, int, int, int) const { return {0.f, 0.f}; }
    __device__ __forceinline__ void operator()(const Feat &, int, int, int, float, float2) const {}
};

}  // namespace dllm
