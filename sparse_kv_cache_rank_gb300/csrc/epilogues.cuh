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
// The GEMM resolves (b, pos) once per token column (pos < 0: not live) and passes
// it with every call; epilogues with kSel == false ignore it.  pre() is the one
// global value an epilogue reads per output (residual input, h1); the GEMM issues
// it for a batch of columns before consuming any, so those loads overlap.
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

// out[m, f] = acc (fp32), for f < n_valid.  Singular proxy and plain GEMM.
struct EpiStoreF32 {
    static constexpr bool kSel = false;
    SelRows sel;
    float *out;
    int ld, n_valid;
    __device__ __forceinline__ float pre(int, int, int, int) const { return 0.f; }
    __device__ __forceinline__ void operator()(int f, int m, int, int, float acc, float) const {
        if (f < n_valid) out[(size_t)m * ld + f] = acc;
    }
};

// [Q | K | V] rows -> rotary embedding at the token's position; Q to the compact
// query buffer, K and V scattered into the cache rows.  rope_cs [M, hd/2] holds
// (cos, sin) of pos * theta^(-2i/hd) for every selected row (written by the gather).
template <class T>
struct EpiQKV {
    static constexpr bool kSel = true;
    SelRows sel;
    T *Q;               // [M, n_q*hd]
    T *Kc, *Vc;         // [B, N, n_kv, hd]
    const float2 *rope_cs;
    int n_q, n_kv, hd, use_rope;

    __device__ __forceinline__ float pre(int, int, int, int) const { return 0.f; }
    __device__ __forceinline__ void operator()(int f, int m, int b, int pos, float acc, float) const {
        const float partner = __shfl_xor_sync(0xffffffffu, acc, 1);
        const int dq = n_q * hd, dkv = n_kv * hd;
        int region, g;
        if (f < dq) { region = 0; g = f; }
        else if (f < dq + dkv) { region = 1; g = f - dq; }
        else { region = 2; g = f - dq - dkv; }
        const int head = g / hd, p = g - head * hd;
        const int i = p >> 1, odd = p & 1;
        const int dim = odd ? i + (hd >> 1) : i;
        float out = acc;
        if (use_rope && region < 2) {
            const float2 cs = rope_cs[(size_t)m * (hd >> 1) + i];
            out = odd ? (acc * cs.x + partner * cs.y) : (acc * cs.x - partner * cs.y);
        }
        if (region == 0) {
            Q[(size_t)m * dq + (size_t)head * hd + dim] = from_f32<T>(out);
        } else if (pos >= 0) {
            T *dst = region == 1 ? Kc : Vc;
            dst[(((size_t)b * sel.N + pos) * n_kv + head) * hd + dim] = from_f32<T>(out);
        }
    }
};

// h1[m, f] = H_in[b, pos, f] + acc (fp32); 0 for rows that are not live.
template <class T>
struct EpiResidual {
    static constexpr bool kSel = true;
    SelRows sel;
    float *h1;          // [M, d]
    const T *H_in;      // [B, N, d]
    int d;
    __device__ __forceinline__ float pre(int f, int, int b, int pos) const {
        return pos >= 0 ? to_f32<T>(H_in[((size_t)b * sel.N + pos) * d + f]) : 0.f;
    }
    __device__ __forceinline__ void operator()(int f, int m, int, int pos, float acc, float hin) const {
        h1[(size_t)m * d + f] = pos >= 0 ? hin + acc : 0.f;
    }
};

// Rows 2j (gate) and 2j+1 (up): U[m, j] = SiLU(gate) * up.
template <class T>
struct EpiSwiGLU {
    static constexpr bool kSel = false;
    SelRows sel;
    T *U;               // [M, F]
    int F;
    __device__ __forceinline__ float pre(int, int, int, int) const { return 0.f; }
    __device__ __forceinline__ void operator()(int f, int m, int, int, float acc, float) const {
        const float partner = __shfl_xor_sync(0xffffffffu, acc, 1);
        if ((f & 1) == 0) U[(size_t)m * F + (f >> 1)] = from_f32<T>(silu(acc) * partner);
    }
};

// H_out_cache[b, pos, f] = h1[m, f] + acc for live rows.
template <class T>
struct EpiDownScatter {
    static constexpr bool kSel = true;
    SelRows sel;
    T *H_out;           // [B, N, d]
    const float *h1;    // [M, d]
    int d;
    __device__ __forceinline__ float pre(int f, int m, int, int pos) const {
        return pos >= 0 ? h1[(size_t)m * d + f] : 0.f;
    }
    __device__ __forceinline__ void operator()(int f, int, int b, int pos, float acc, float h) const {
        if (pos >= 0) H_out[((size_t)b * sel.N + pos) * d + f] = from_f32<T>(h + acc);
    }
};

}  // namespace dllm
