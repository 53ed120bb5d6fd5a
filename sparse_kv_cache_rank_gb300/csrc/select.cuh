// select.cuh -- the per-sequence selection of the drift top-k united with the forced
// rows (SPA-Cache, "1. Update identification via singular proxy", "2. Adaptive budget
// allocation"; EntropyCache, "How EntropyCache works", step 3), as a block-level device
// function shared by the selection kernel and the fused selection + gather kernel.
//
// The k-th largest drift is found exactly by a radix select on order-preserving 32-bit
// keys (up to 4 passes of 256-bin shared histograms); rows above it are taken, rows equal
// to it are taken in index order until the budget is met (lower row index wins ties), and
// the union with the forced rows is compacted in ascending order by a block-wide scan.
// The passes stop early once the digit holding the k-th key is taken whole: every key
// from that digit's lower bound up is then selected and no tie needs ranking.
#pragma once

#include "internal.h"

namespace dllm {

// Exclusive block scan of one value per thread; returns the exclusive prefix and
// writes the block total to *total.  All threads must call it.
template <int kT>
__device__ __forceinline__ uint32_t block_scan(uint32_t v, uint32_t *wsum, uint32_t *total) {
    constexpr int kWarps = kT / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < kWarps ? wsum[lane] : 0u;
        uint32_t s = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        wsum[lane] = s - w;   // exclusive prefix of the warp totals
        if (lane == 31) wsum[32] = s;
    }
    __syncthreads();
    const uint32_t r = wsum[warp] + x - v;
    *total = wsum[32];
    __syncthreads();
    return r;
}

// Selection of one sequence by the whole block (kT threads): key [N] and flag [N] are
// shared-memory scratch; out[0 .. total) receives the selected rows in ascending order and
// out[total .. N) = -1 (out may be global or shared memory).  Returns total.  N < 65536.
template <int kT>
__device__ uint32_t select_sequence(const float *__restrict__ dr, const int32_t *__restrict__ forced_b, int F,
                                    int k, float min_drift, int N, uint32_t *key, uint8_t *flag, int32_t *out) {
    __shared__ uint32_t hist[256];
    __shared__ uint32_t wsum[33];
    __shared__ uint32_t sh_prefix, sh_rem, sh_whole;
    const int tid = threadIdx.x;
    for (int i = tid; i < N; i += kT) flag[i] = 0;
    __syncthreads();
    if (forced_b)
        for (int f = tid; f < F; f += kT) {
            const int p = forced_b[f];
            if (p >= 0 && p < N) flag[p] = 1;
        }
    __syncthreads();

    // contiguous chunk per thread keeps index order for the scans below
    const int C = (N + kT - 1) / kT;
    const int i0 = min(N, tid * C), i1 = min(N, i0 + C);
    uint32_t nf = 0, ne = 0;
    for (int i = i0; i < i1; ++i) {
        uint32_t kk = 0;
        const float x = __ldcg(dr + i);   // L2: the drifts may have been written by other CTAs
        if (flag[i]) {
            ++nf;
        } else if (x > min_drift) {   // false for NaN
            const uint32_t u = __float_as_uint(x);
            kk = (u & 0x80000000u) ? ~u : (u | 0x80000000u);   // order-preserving, > 0
            ++ne;
        }
        key[i] = kk;
    }
    uint32_t tot_fe;   // both counts in one scan (N <= 16384 < 2^16)
    block_scan<kT>((nf << 16) | ne, wsum, &tot_fe);
    const uint32_t tot_f = tot_fe >> 16, tot_e = tot_fe & 0xFFFFu;
    long long budget = (long long)N - tot_f;
    if ((long long)k < budget) budget = k;
    if (budget < 0) budget = 0;
    const uint32_t take = (uint32_t)(budget < (long long)tot_e ? budget : (long long)tot_e);

    // threshold T: take every key > T and the first `rem` keys == T (index order)
    uint32_t T, rem;
    if (take == 0) {
        T = 0xFFFFFFFFu;
        rem = 0;
    } else if (take == tot_e) {
        T = 0;
        rem = 0;
    } else {
        uint32_t prefix = 0, mask = 0;
        bool whole = false;
        rem = take;
        for (int shift = 24; shift >= 0 && !whole; shift -= 8) {
            for (int i = tid; i < 256; i += kT) hist[i] = 0;
            __syncthreads();
            // warp-aggregated counts: most keys share their leading digits, so one
            // atomic per distinct digit per warp instead of one per key
            for (int c = 0; c < C; ++c) {
                const int i = i0 + c;
                uint32_t dg = 256u;   // no digit
                if (i < i1) {
                    const uint32_t kk = key[i];
                    if (kk != 0 && (kk & mask) == prefix) dg = (kk >> shift) & 255u;
                }
                const uint32_t same = __match_any_sync(0xffffffffu, dg);
                if (dg < 256u && (threadIdx.x & 31) == __ffs(same) - 1) atomicAdd(&hist[dg], (uint32_t)__popc(same));
            }
            __syncthreads();
            if (tid < 32) {
                // lane l owns digits 255-8l .. 248-8l (descending); suffix counts by a
                // warp scan find the digit holding the rem-th largest key
                uint32_t h[8], own = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    h[j] = hist[255 - 8 * tid - j];
                    own += h[j];
                }
                uint32_t incl = own;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (tid >= o) incl += y;
                }
                uint32_t cum = incl - own;   // keys in higher digits than this lane's
                if (cum < rem && rem <= incl) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        if (cum + h[j] >= rem) {
                            sh_prefix = prefix | ((uint32_t)(255 - 8 * tid - j) << shift);
                            sh_rem = rem - cum;
                            sh_whole = cum + h[j] == rem;   // the digit's keys are all taken
                            break;
                        }
                        cum += h[j];
                    }
                }
            }
            __syncthreads();
            prefix = sh_prefix;
            rem = sh_rem;
            whole = sh_whole != 0;
            mask |= 255u << shift;
            __syncthreads();
        }
        if (whole) {   // take every key >= the digit's lower bound (prefix, low bits 0)
            T = prefix ? prefix - 1u : 0u;
            rem = 0;
        } else {
            T = prefix;
        }
    }

    // rank of each key == T among equals, in index order (rem is the same in every thread:
    // no ranking, and no scan, when no tie straddles the budget)
    uint32_t eq_before = 0;
    if (rem > 0) {
        uint32_t neq = 0, tot_eq;
        for (int i = i0; i < i1; ++i) neq += (key[i] == T);
        eq_before = block_scan<kT>(neq, wsum, &tot_eq);
    }
    uint32_t nsel = 0;
    for (int i = i0; i < i1; ++i) {
        const uint32_t kk = key[i];
        bool s = flag[i] != 0 || (kk != 0 && kk > T);
        if (!s && rem > 0 && kk == T && kk != 0) {
            s = eq_before < rem;
            ++eq_before;
        }
        flag[i] = s ? 2 : 0;
        nsel += s;
    }
    uint32_t total;
    uint32_t o = block_scan<kT>(nsel, wsum, &total);
    for (int i = i0; i < i1; ++i)
        if (flag[i] == 2) out[o++] = i;
    for (int i = (int)total + tid; i < N; i += kT) out[i] = -1;
    __syncthreads();
    return total;
}

}  // namespace dllm
