// gemm_tc.cu -- weight-stationary bf16 GEMM on the sm_103a tensor cores
// (tcgen05.mma, fp32 accumulators in TMEM, operands staged by TMA).
//
// acc[f, m] = <W[f, :], X[m, :]>: the weight tile (128 rows of W) is the MMA's
// A operand (M = 128) and a tile of BN token rows is its B operand (N = BN), so a
// GEMM over few gathered tokens (the selected rows) wastes no MMA rows on padding.
// Each CTA owns one (weight tile, token tile) pair, and, when the tiles alone cannot
// fill the GPU, one K slice of it: the CTAs of one K split form a thread-block
// cluster and reduce their fp32 partial tiles through distributed shared memory.
// Weight bytes are read from HBM once (token tiles of one weight tile run side by
// side and share it through L2).
//
// Roles (64 + 32 EW threads):  warp 0 lane 0   TMA producer (multi-stage ring)
//                              warp 1          TMEM owner; lane 0 issues the MMAs
//                              warps 2..EW+1   epilogue, EW / 4 warps per TMEM lane
//                                              quarter, each taking a share of the token
//                                              columns (EW = 8 at two CTAs per SM, 16 at
//                                              one: the epilogue after a K split's main
//                                              loop is a chain of dependent loads)
// Without a K split the epilogue reads the accumulator straight from TMEM and the
// CTA needs no shared memory beyond the ring, so two CTAs fit on an SM and one
// CTA's epilogue overlaps the other's main loop.
#include <cudaTypedefs.h>

#include <mutex>
#include <type_traits>

#include "internal.h"

namespace dllm {
namespace {

constexpr int BM = 128;                // weight rows per tile (MMA M)
constexpr int BK = 64;                 // K per stage: one 128-byte swizzled row of bf16
constexpr int kWBytes = BM * BK * 2;   // 16 KB
constexpr int kSmemLimit = 232448;     // 227 KB dynamic shared memory per CTA
constexpr int kSmemPair = 113 * 1024;  // budget per CTA when two share an SM
constexpr int kGroupW = 16;            // weight tiles per group of the tile order
constexpr int kTailBytes = 256;        // barriers, TMEM slot, abort flag
                                       // then per token column (sequence, position): 8 * BN bytes

struct Shape {
    int M_tok, N_out, K;
    int BN, splits, stages;
    int w_const;      // weights are never written on the device: stream them before the wait
    int indep;        // K slices are independent CTAs (no cluster): slice z writes token rows
                      // z * M_tok + m of the epilogue's output (partial sums, reduced later)
    int body_bytes;   // pipeline ring (and, with a cluster K split, the fp32 partial tile [BN][128])
    int xrows;        // token rows staged per K block (<= BN; the MMA's N = BN columns past xrows
                      // read whatever follows in shared memory and are never stored)
    int base_aligned; // no alignment slack was reserved: the dynamic shared memory must start
                      // on a 1024-byte boundary (else the kernel reports it and does nothing)
    int col_bytes;    // per token column (sequence, position) after the body, >= 8 * BN and
                      // >= the bytes the MMA reads past the last stage; barriers follow
    int w_stream;     // the weights are larger than a fraction of L2 and read once per call:
                      // their lines are loaded with an evict-first policy
    unsigned *zero;   // nzero words the first CTA clears once the previous kernel is done
    int nzero;        // (counters of the kernel that follows; nullptr / 0: none)
};

__host__ __device__ inline int stage_bytes(int xrows) { return kWBytes + xrows * BK * 2; }

// Applies the epilogue to 16 consecutive token columns c0.. of feature row F held in
// v[]: the global values of all 16 outputs are requested before the first is written.
template <class Epi>
__device__ __forceinline__ void epi_16(const Epi &epi, const typename Epi::Feat &F, int m0, int c0,
                                       int ncols, const int *col_b, const int *col_pos,
                                       const float (&v)[16]) {
    float2 pr[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int cc = min(c0 + j, ncols - 1);
        pr[j] = epi.pre(F, m0 + cc, col_b[cc], col_pos[cc]);
    }
#pragma unroll
    for (int j = 0; j < 16; ++j)
        if (c0 + j < ncols) epi(F, m0 + c0 + j, col_b[c0 + j], col_pos[c0 + j], v[j], pr[j]);
}

// Epilogues that reduce over the tile's features (EpiCosine) declare kCosine = true.
template <class E, class = void>
struct epi_cosine : std::false_type {};
template <class E>
struct epi_cosine<E, std::void_t<decltype(E::kCosine)>> : std::integral_constant<bool, E::kCosine> {};

// Scratch of the feature reduction per share of columns: [4 quarters][32] squared norms,
// then [4 quarters][16] squared differences.
constexpr int kCosRed = 4 * 32 + 4 * 16;

// Warp reduce-scatter of 2W values: afterwards v[0] of lane l holds the warp's sum of
// value (l & (2W - 1)) (rounds over lane bits log2(W) .. 0; lanes that differ only above
// them hold the same sums when every lane starts with the same set).
template <int W>
__device__ __forceinline__ void warp_reduce_scatter(float (&v)[2 * W], int lane) {
#pragma unroll
    for (int w = W; w >= 1; w >>= 1) {
        const bool up = (lane & w) != 0;
#pragma unroll
        for (int i = 0; i < w; ++i) {
            const float send = up ? v[i] : v[i + w];
            const float keep = up ? v[i + w] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
        }
    }
}

// Barrier of the four warps of column share `part` (ids 2..5, immediates so that the
// kernel reserves only the barriers it names).
__device__ __forceinline__ void share_bar(int part) {
    __syncwarp();
    switch (part) {
        case 0: asm volatile("bar.sync 2, 128;" ::: "memory"); break;
        case 1: asm volatile("bar.sync 3, 128;" ::: "memory"); break;
        case 2: asm volatile("bar.sync 4, 128;" ::: "memory"); break;
        default: asm volatile("bar.sync 5, 128;" ::: "memory"); break;
    }
}

// Cosine drift of token columns c0 .. c0+15 (live below cend) of a tile whose thread holds
// feature f = 32 q + lane of each column in acc[].  The four warps of one share of the
// columns (one per TMEM lane quarter) call this together.
template <class Epi>
__device__ __forceinline__ void cosine_16(const Epi &epi, int f, int q, int lane, int m0, int c0, int cend,
                                          const float (&acc)[16], float *red, int part) {
    const bool fv = f < epi.r;
    float a[16], cv[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const bool live = fv && c0 + j < cend;
        const size_t o = (size_t)(m0 + c0 + j) * (size_t)epi.r + (size_t)f;
        a[j] = live ? acc[j] : 0.f;
        cv[j] = live ? __ldcg(epi.cached + o) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j)
        if (fv && c0 + j < cend) epi.cur[(size_t)(m0 + c0 + j) * (size_t)epi.r + (size_t)f] = a[j];
    // squared norms: lane l of quarter q ends with column (l & 15)'s sum over the
    // quarter's 32 features, of the current proxy (l < 16) or the cached one
    float v[32];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        v[j] = a[j] * a[j];
        v[16 + j] = cv[j] * cv[j];
    }
    warp_reduce_scatter<16>(v, lane);
    red[q * 32 + lane] = v[0];
    share_bar(part);
    float na[16], nc[16], t[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        na[j] = ((red[j] + red[32 + j]) + red[64 + j]) + red[96 + j];
        nc[j] = ((red[16 + j] + red[48 + j]) + red[80 + j]) + red[112 + j];
        float d = 0.f;
        if (na[j] != 0.f && nc[j] != 0.f) {
            const float ia = 1.0f / sqrtf(na[j]), ic = 1.0f / sqrtf(nc[j]);
            // separately rounded products (no FMA contraction): equal inputs give d == 0
            d = __fsub_rn(__fmul_rn(a[j], ia), __fmul_rn(cv[j], ic));
        }
        t[j] = d * d;
    }
    // the squared differences: both lane halves hold the same 16 sums after the
    // exchange across lane bit 4, then lane l holds column (l & 15)'s quarter sum
#pragma unroll
    for (int j = 0; j < 16; ++j) t[j] += __shfl_xor_sync(0xffffffffu, t[j], 16);
    warp_reduce_scatter<8>(t, lane);
    if (lane < 16) red[128 + q * 16 + lane] = t[0];
    share_bar(part);
    if (q == 0 && lane < 16 && c0 + lane < cend) {
        float n_a = 0.f, n_c = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (j == lane) {
                n_a = na[j];
                n_c = nc[j];
            }
        float out;
        if (n_a == 0.f && n_c == 0.f) {
            out = 0.f;
        } else if (n_a == 0.f || n_c == 0.f) {
            out = 1.f;
        } else {
            const float sd = ((red[128 + lane] + red[144 + lane]) + red[160 + lane]) + red[176 + lane];
            out = fminf(fmaxf(0.5f * sd, 0.f), 2.f);
        }
        epi.drift[m0 + c0 + lane] = out;
    }
}

template <class Epi, int EW>
__global__ void __launch_bounds__(64 + 32 * EW, EW == 8 ? 2 : 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
              const Shape g, const Epi epi, unsigned *status) {
    constexpr int NP = EW / 4;   // epilogue warps per TMEM lane quarter
    constexpr bool kCos = epi_cosine<Epi>::value;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;   // 1024-byte aligned: required by the 128-byte swizzle
    if (g.base_aligned && pad != 0) {  // the plan left no room to align: do nothing, loudly
        griddep_wait();
        if (threadIdx.x == 0) raise_status(status, DLLM_STATUS_SMEM_LAYOUT);
        return;
    }
    int *col_b = reinterpret_cast<int *>(smem + g.body_bytes);   // [BN] then col_pos [BN]
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + g.body_bytes + g.col_bytes);
    uint64_t *empty = full + g.stages;
    uint64_t *done = empty + g.stages;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *col_pos = col_b + g.BN;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // tile order: with several token tiles, consecutive CTAs walk groups of kGroupW
    // weight tiles one token tile at a time, so that the tiles resident at once share few
    // weight and token tiles and their re-reads hit L2 (the plain order would stream every
    // token tile past every weight tile from HBM once the token rows outgrow L2)
    int tt = blockIdx.x, wt = blockIdx.y;
    if (gridDim.x > 1) {
        const int lin = blockIdx.y * gridDim.x + blockIdx.x;
        const int per_group = kGroupW * gridDim.x;
        const int first_w = lin / per_group * kGroupW;
        const int gsize = min((int)gridDim.y - first_w, kGroupW);
        const int in_group = lin - (first_w / kGroupW) * per_group;
        wt = first_w + in_group % gsize;
        tt = in_group / gsize;
    }
    const int m0 = tt * g.BN;
    const int n0 = wt * BM;
    const int split = g.indep ? (int)blockIdx.z : (g.splits > 1 ? (int)cluster_ctarank() : 0);
    const bool cluster_split = g.splits > 1 && !g.indep;
    const int KB = g.K / BK;
    const int kb0 = (int)((long long)split * KB / g.splits);
    const int kb1 = (int)((long long)(split + 1) * KB / g.splits);
    const int nkb = kb1 - kb0;
    const uint32_t tmem_cols = g.BN <= 32 ? 32u : g.BN <= 64 ? 64u : g.BN <= 128 ? 128u : 256u;
    const int sbytes = stage_bytes(g.xrows);
    const int ncols = min(g.BN, g.M_tok - m0);   // live token columns of this tile

    if (threadIdx.x == 0) {
        for (int s = 0; s < g.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmW);
        tma_prefetch_desc(&tmX);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, tmem_cols);
        tmem_relinquish();
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    griddep_launch();
    if (warp == 0) {
        if (lane == 0) {   // ---------------- TMA producer
            // weights never change on the device: the first ring stages stream their
            // weight tiles while the previous kernel is still draining
            const uint64_t pol = l2_policy_evict_first();
            auto load_w = [&](void *dst, uint64_t *bar, int kb) {
                if (g.w_stream) tma_load_2d_hint(dst, &tmW, bar, kb * BK, n0, pol);
                else tma_load_2d(dst, &tmW, bar, kb * BK, n0);
            };
            const int pre = g.w_const ? (nkb < g.stages ? nkb : g.stages) : 0;
            for (int it = 0; it < pre; ++it) {
                mbar_arrive_expect_tx(&full[it], (uint32_t)sbytes);
                load_w(smem + it * sbytes, &full[it], kb0 + it);
            }
            griddep_wait();
            for (int it = 0; it < pre; ++it)
                tma_load_2d(smem + it * sbytes + kWBytes, &tmX, &full[it], (kb0 + it) * BK, m0);
            int issued = pre;
            for (int it = pre; it < nkb; ++it) {
                const int s = it % g.stages;
                const uint32_t ph = (uint32_t)(it / g.stages) & 1u;
                if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, status)) break;
                uint8_t *sw = smem + s * sbytes;
                mbar_arrive_expect_tx(&full[s], (uint32_t)sbytes);
                load_w(sw, &full[s], kb0 + it);
                tma_load_2d(sw + kWBytes, &tmX, &full[s], (kb0 + it) * BK, m0);
                ++issued;
            }
            if (*abort_flag) {   // every issued copy must land before the CTA can exit
                for (int it = issued > g.stages ? issued - g.stages : 0; it < issued; ++it)
                    mbar_drain(&full[it % g.stages], (uint32_t)(it / g.stages) & 1u);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {   // ---------------- MMA issuer
            const uint32_t idesc = idesc_bf16(BM, g.BN, 0);
            for (int it = 0; it < nkb; ++it) {
                const int s = it % g.stages;
                const uint32_t ph = (uint32_t)(it / g.stages) & 1u;
                if (!mbar_wait(&full[s], ph, abort_flag, status)) break;
                tc_fence_after();
                const uint32_t aw = smem_u32(smem + s * sbytes);
                const uint32_t ax = aw + kWBytes;
#pragma unroll
                for (int k = 0; k < BK / 16; ++k)   // K = 16 per MMA: +32 bytes inside the swizzle row
                    mma_bf16(tmem, smem_desc_sw128(aw + k * 32, 16, 1024),
                             smem_desc_sw128(ax + k * 32, 16, 1024), idesc, (it | k) != 0);
                mma_commit(&empty[s]);   // frees the stage once these MMAs have read it
            }
            mma_commit(done);
        }
    } else {
        // ---------------- epilogue warps (2..9): resolve every token column's (sequence,
        // position) while the main loop runs
        griddep_wait();
        if (g.zero && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
            for (int i = threadIdx.x - 64; i < g.nzero; i += 32 * EW) g.zero[i] = 0u;
        for (int c = threadIdx.x - 64; c < (kCos ? 0 : g.BN); c += 32 * EW) {
            int b = 0, pos = -1;
            if constexpr (Epi::kColScale) {   // a per-column scale in the position slot
                col_b[c] = 0;
                col_pos[c] = __float_as_int(c < ncols ? epi.col_scale(m0 + c) : 0.f);
                continue;
            }
            if (Epi::kSel && c < ncols) epi.sel.locate(m0 + c, b, pos);
            col_b[c] = b;
            col_pos[c] = pos;
        }
        __syncwarp();
        named_bar_sync(1, EW * 32);
        mbar_wait(done, 0, abort_flag, status);
        tc_fence_after();
        const int q = warp & 3;                  // TMEM lane quarter this warp may access
        const int part = (warp - 2) >> 2;        // which share of the columns
        const int f = q * 32 + lane;
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16);
        const int nchunk = (g.BN + 15) / 16;
        const int ch0 = part * nchunk / NP, ch1 = (part + 1) * nchunk / NP;
        if constexpr (Epi::kTileReduce) {
            // one softmax state per token column over this tile's 128 weight rows: a
            // butterfly over the 32 rows of each warp, then the 4 lane quarters in order
            // (the ring is idle once `done` has completed)
            VocabState *red = reinterpret_cast<VocabState *>(smem);   // [4][BN]
            const bool rows_ok = n0 + q * 32 < g.N_out;                // warp-uniform
            for (int ch = ch0; ch < ch1; ++ch) {
                float v[16];
                tmem_ld_x16(taddr + (uint32_t)(ch * 16), v);
                tmem_ld_wait(v);
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    VocabState st = rows_ok ? VocabState{v[j], 1.f, 0.f, n0 + f}
                                            : VocabState{-INFINITY, 0.f, 0.f, INT_MAX};
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        VocabState y;
                        y.m = __shfl_xor_sync(0xffffffffu, st.m, o);
                        y.s = __shfl_xor_sync(0xffffffffu, st.s, o);
                        y.t = __shfl_xor_sync(0xffffffffu, st.t, o);
                        y.a = __shfl_xor_sync(0xffffffffu, st.a, o);
                        st = (lane & o) ? vocab_merge(y, st) : vocab_merge(st, y);
                    }
                    if (lane == 0) red[q * g.BN + ch * 16 + j] = st;
                }
            }
            __syncwarp();
            named_bar_sync(1, EW * 32);
            for (int c = threadIdx.x - 64; c < ncols; c += EW * 32) {
                VocabState r = red[c];
#pragma unroll
                for (int qq = 1; qq < 4; ++qq) r = vocab_merge(r, red[qq * g.BN + c]);
                epi.part[(size_t)(m0 + c) * epi.tiles + wt] = r;
            }
        } else if (kCos) {
            // the drift of each token column straight from TMEM (no K split: the planner
            // gives EpiCosine one CTA per token tile; the scratch follows the ring, in the
            // per-column area this epilogue does not use)
            float *red = reinterpret_cast<float *>(smem + g.body_bytes) + part * kCosRed;
            for (int ch = ch0; ch < ch1 && ch * 16 < ncols; ++ch) {
                float v[16];
                tmem_ld_x16(taddr + (uint32_t)(ch * 16), v);
                tmem_ld_wait(v);
                if constexpr (kCos) cosine_16(epi, f, q, lane, m0, ch * 16, ncols, v, red, part);
            }
        } else if (!cluster_split) {
            // straight from TMEM (independent K slices write rows split * M_tok + m)
            const int moff = g.indep ? split * g.M_tok : 0;
            if (n0 + q * 32 < g.N_out) {   // warp-uniform: N_out % 32 == 0
                const typename Epi::Feat F = epi.feat(n0 + f);
                for (int ch = ch0; ch < ch1 && ch * 16 < ncols; ++ch) {
                    float v[16];
                    tmem_ld_x16(taddr + (uint32_t)(ch * 16), v);
                    tmem_ld_wait(v);
                    epi_16(epi, F, m0 + moff, ch * 16, ncols, col_b, col_pos, v);
                }
            }
        } else {
            // K split: fp32 partial tile [BN][128] into this CTA's shared memory
            float *part = reinterpret_cast<float *>(smem);
            for (int ch = ch0; ch < ch1; ++ch) {
                float v[16];
                tmem_ld_x16(taddr + (uint32_t)(ch * 16), v);
                tmem_ld_wait(v);
#pragma unroll
                for (int j = 0; j < 16; ++j) part[(ch * 16 + j) * BM + f] = v[j];
            }
        }
    }
    __syncwarp();   // each warp converged before the block-wide / cluster-wide barrier
    tc_fence_before();
    if (cluster_split) {
        cluster_sync_all();
        if (warp >= 2) {   // ---------------- reduce the cluster's partials, epilogue on my share
            const int q = warp & 3;
            const int part = (warp - 2) >> 2;
            const int f = q * 32 + lane;
            const int per = (((g.BN + g.splits - 1) / g.splits) + 15) / 16 * 16;
            const int cb = split * per;
            const int ce = min(min(g.BN, cb + per), ncols);
            const int pper = (((ce - cb) + NP - 1) / NP + 15) / 16 * 16;   // 16-column aligned shares
            const int c_begin = min(ce, cb + part * pper);
            const int c_end = part == NP - 1 ? ce : min(ce, cb + (part + 1) * pper);
            const uint32_t part_s = smem_u32(smem) + (uint32_t)f * 4u;
            if (n0 + q * 32 < g.N_out) {
                const typename Epi::Feat F = epi.feat(n0 + f);
                for (int c = c_begin; c < c_end; c += 16) {
                    float acc[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) acc[j] = 0.f;
                    // two CTAs' columns in flight at once, added in rank order
                    for (int r = 0; r < g.splits; r += 2) {
                        const bool two = r + 1 < g.splits;
                        const uint32_t ba = mapa_shared(part_s, (uint32_t)r);
                        const uint32_t bb = mapa_shared(part_s, (uint32_t)(two ? r + 1 : r));
                        float va[16], vb[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const uint32_t off = (uint32_t)(min(c + j, c_end - 1) * BM) * 4u;
                            va[j] = ld_dsmem_f32(ba + off);
                            vb[j] = ld_dsmem_f32(bb + off);
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j) acc[j] += va[j];
                        if (two) {
#pragma unroll
                            for (int j = 0; j < 16; ++j) acc[j] += vb[j];
                        }
                    }
                    epi_16(epi, F, m0, c, c_end, col_b, col_pos, acc);
                }
            }
        }
        __syncwarp();
        cluster_sync_all();   // peers may still read this CTA's partial tile
    } else {
        __syncthreads();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, tmem_cols);
    }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace

// Row-major bf16 matrix [rows, cols], boxes of 64 columns x box_rows rows, 128-byte swizzle.
// Encoded maps are cached per host thread (a step re-encodes the same few operands
// every call; the descriptor depends only on these four values and the device).
bool make_tmap(CUtensorMap *tm, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    struct Entry {
        const void *base;
        uint64_t rows, cols;
        uint32_t box_rows;
        int dev;
        CUtensorMap map;
    };
    constexpr int kSlots = 64;
    thread_local Entry cache[kSlots] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t h = (reinterpret_cast<uint64_t>(base) >> 8) ^ (rows * 0x9E3779B97F4A7C15ull) ^
                       (cols << 7) ^ ((uint64_t)box_rows << 3) ^ (uint64_t)dev;
    Entry &e = cache[(h ^ (h >> 29)) % kSlots];
    if (e.base == base && e.rows == rows && e.cols == cols && e.box_rows == box_rows && e.dev == dev &&
        base != nullptr) {
        *tm = e.map;
        return true;
    }
    auto enc = tmap_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, box_rows};
    cuuint32_t estr[2] = {1, 1};
    if (enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    e.base = base;
    e.rows = rows;
    e.cols = cols;
    e.box_rows = box_rows;
    e.dev = dev;
    e.map = *tm;
    return true;
}

namespace {

struct Plan {
    int BN, splits, stages, tok_tiles, w_tiles;
    int body, xrows, base_aligned, col_bytes;
    size_t smem;
};

int round16(int x) { return (x + 15) / 16 * 16; }

Plan make_plan(int M_tok, int N_out, int K, int BN, int splits, int budget, bool smem_partial,
               int min_col_bytes = 0) {
    Plan p{};
    p.BN = BN;
    p.splits = splits;
    p.w_tiles = (N_out + BM - 1) / BM;
    p.tok_tiles = (M_tok + BN - 1) / BN;
    // one token tile: stage only the rows that exist, rounded up to the 8-row swizzle atom
    const int r8 = (M_tok + 7) / 8 * 8;
    p.xrows = p.tok_tiles == 1 && r8 < BN ? r8 : BN;
    const int sb = stage_bytes(p.xrows);
    const int over = (BN - p.xrows) * BK * 2;   // read by the MMA past the last stage
    p.col_bytes = 8 * BN > over ? 8 * BN : over;
    if (p.col_bytes < min_col_bytes) p.col_bytes = min_col_bytes;
    const int tail = p.col_bytes + kTailBytes;
    const int part = smem_partial ? BN * BM * 4 : 0;
    const int KB = K / BK;
    auto fit = [&](int slack) {
        int st = (budget - slack - tail) / sb;
        if (st > 8) st = 8;
        if (st > KB / splits + 1) st = KB / splits + 1 > 2 ? KB / splits + 1 : 2;
        return st;
    };
    p.stages = fit(1024);
    p.base_aligned = 0;
    // one stage more when only the 1 KB alignment slack stands in the way.  The offset of
    // dynamic shared memory is the same in every CTA of a launch, so a misaligned base
    // sends every CTA of a cluster back before its first cluster barrier, together.
    if (fit(0) > p.stages) {
        p.stages = fit(0);
        p.base_aligned = 1;
    }
    p.body = p.stages * sb > part ? p.stages * sb : part;
    p.smem = (size_t)(p.base_aligned ? 0 : 1024) + p.body + tail;
    return p;
}

// Token-tile width (and K split) for many tokens (M > 256).  A CTA here is latency-bound:
// its time per K block barely changes whether it shares the SM or not, and it depends on
// the width mostly through the pipeline depth that two CTAs per SM leave (three stages up
// to 160 columns, two above).  So a width is charged, per round of two CTAs on every SM, a
// fixed cost plus K blocks x its time per K block; a last round of at most one CTA per SM
// takes the time of a CTA alone.  The times are least-squares fits to the layer
// projections of a GB300 over N = 2048..8192 tokens (LLaDA-8B and Dream-7B shapes), where
// the model picks the fastest width in 19 of 20 cases.  A K split over a cluster divides a
// CTA's K blocks and multiplies the CTAs (considered when the fp32 partial tile still fits
// two CTAs per SM), for a fixed reduction cost; it pays where the tiles alone leave a round
// far from full.  Returns 0 when no plan gives at least half the SMs a CTA.
int pick_bn_many(int M_tok, int w_tiles, int KB, int sms, int *splits) {
    static const int bns[] = {128, 160, 176, 192, 208, 224, 256};
    static const float us_pair[] = {0.378f, 0.433f, 0.592f, 0.616f, 0.652f, 0.688f, 0.758f};
    static const float us_alone[] = {0.311f, 0.388f, 0.617f, 0.625f, 0.660f, 0.647f, 0.690f};
    const float us_fixed = 14.6f, us_split = 2.0f;
    const long long slots = 2LL * sms;
    int best = 0, best_s = 1;
    float best_us = 0.f;
    for (int i = 0; i < 7; ++i) {
        const long long tiles = (long long)w_tiles * ((M_tok + bns[i] - 1) / bns[i]);
        const bool pair_split = bns[i] * BM * 4 + 1024 + kTailBytes + 8 * bns[i] <= kSmemPair;
        for (int s = 1; s <= 8; ++s) {
            if (s > 1 && (!pair_split || KB / s < 2)) break;
            const long long ctas = tiles * s;
            if (2 * ctas < sms) continue;
            const long long rounds = (ctas + slots - 1) / slots;
            const long long last = ctas - slots * (rounds - 1);
            const float kb = (float)KB / (float)s;
            const float us = (float)(rounds - 1) * (us_fixed + kb * us_pair[i]) + us_fixed +
                             kb * (last <= sms ? us_alone[i] : us_pair[i]) + (s > 1 ? us_split : 0.f);
            if (best == 0 || us < best_us) {
                best = bns[i];
                best_s = s;
                best_us = us;
            }
        }
    }
    *splits = best_s;
    return best;
}

// Few tokens (the gathered rows of a step) make every projection a weight stream:
// what matters is that every SM streams weights and that epilogues overlap main loops.
//  * many weight tiles (>= half the SMs): two CTAs per SM; no K split when the weight
//    tiles fill the SMs, else a K split over a cluster sized to about two CTAs per SM;
//  * few weight tiles: a K split across a cluster sized to fill the SMs.
// Many tokens: the token-tile width that the tile-time model below finds fastest, two
// CTAs per SM; a K split only when no width gives half the SMs a tile.
Plan plan_gemm(int M_tok, int N_out, int K, int splits_req, int sms) {
    const int w_tiles = (N_out + BM - 1) / BM;
    const int KB = K / BK;
    auto clamp_splits = [&](int s) {
        s = s < 1 ? 1 : (s > 8 ? 8 : s);
        while (s > 1 && KB / s < 2) --s;
        return s;
    };
    if (splits_req > 0) {
        const int BN = M_tok <= 256 ? round16(M_tok) : 256;
        const int s = clamp_splits(splits_req);
        // two CTAs per SM whenever the fp32 partial tile of a K split fits their share
        const bool pair = s == 1 || BN * BM * 4 + 1024 + kTailBytes + 8 * BN <= kSmemPair;
        return make_plan(M_tok, N_out, K, BN, s, pair ? kSmemPair : kSmemLimit, s > 1);
    }
    if (M_tok <= 256) {
        if (2 * w_tiles >= sms) {
            const int BN = round16(M_tok);
            if (w_tiles < sms && M_tok > 32) {
                // fewer weight tiles than SMs: a K split over a cluster, two CTAs per SM, so
                // that every SM streams weights (each weight byte is still read once)
                int s = clamp_splits(2 * sms / w_tiles);
                s = s > 4 ? 4 : s;
                if (s > 1 && BN * BM * 4 + 1024 + kTailBytes + 8 * BN <= kSmemPair)
                    return make_plan(M_tok, N_out, K, BN, s, kSmemPair, true);
            }
            return make_plan(M_tok, N_out, K, BN, 1, kSmemPair, false);
        }
        int BN = round16(M_tok);
        const int tok_tiles = 1;
        const int s = clamp_splits(sms / (w_tiles * tok_tiles));
        return make_plan(M_tok, N_out, K, BN, s, s == 1 ? kSmemPair : kSmemLimit, s > 1);
    }
    int s_model = 1;
    int BN = pick_bn_many(M_tok, w_tiles, KB, sms, &s_model);
    if (BN != 0 && s_model > 1) return make_plan(M_tok, N_out, K, BN, s_model, kSmemPair, true);
    if (BN == 0) {
        BN = 256;
        while (BN > 64 && (long long)w_tiles * ((M_tok + BN - 1) / BN) * 8 < sms) BN = round16(BN / 2);
    }
    const long long tiles = (long long)w_tiles * ((M_tok + BN - 1) / BN);
    if (tiles >= sms) return make_plan(M_tok, N_out, K, BN, 1, kSmemPair, false);
    // fewer tiles than SMs (a few hundred tokens against a narrow weight, e.g. the O and
    // down projections at 257..600 rows): a K split over a cluster so that every SM
    // streams, two CTAs per SM when the fp32 partial tile fits their share
    const bool pair = BN * BM * 4 + 1024 + kTailBytes + 8 * BN <= kSmemPair;
    const int s = clamp_splits((int)((pair ? 2 : 1) * (long long)sms / tiles));
    return make_plan(M_tok, N_out, K, BN, s, s > 1 && !pair ? kSmemLimit : kSmemPair, s > 1);
}

// Independent K slices (no cluster), each writing its own fp32 partial output: token
// tiles of 64 rows (128 beyond 2048 tokens), slices sized to two CTAs per SM.  (At 1024
// tokens the 128 CTAs fit one per SM; giving each the whole SM's shared memory, so that
// all 8 K blocks of a slice are in flight, measured 1 us slower: 10.8 against 9.9 us.)
Plan plan_slices(int M_tok, int N_out, int K, int sms) {
    const int KB = K / BK;
    const int BN = M_tok <= 256 ? round16(M_tok) : (M_tok <= 2048 ? 64 : 128);
    const long long tiles = (long long)((N_out + BM - 1) / BM) * ((M_tok + BN - 1) / BN);
    int s = (int)(2 * sms / tiles);
    s = s < 1 ? 1 : (s > 8 ? 8 : s);
    while (s > 1 && KB / s < 2) --s;
    return make_plan(M_tok, N_out, K, BN, s, kSmemPair, false);
}

// The proxy projection with its cosine drift in the epilogue (r <= 128: one weight tile
// holds every feature of a token), for the shapes whose slice plan needs no K split (the
// token tiles alone give every SM two CTAs, or K is too short to split): the tiles of
// plan_slices, one CTA each.  The per-column area after the ring holds the epilogue's
// feature-reduction scratch.  (Split shapes keep the slices and the cosine kernel: a K
// split reduced inside 8-CTA clusters measured 24.5 us against 9.9 + 4.3 us at 1024
// tokens, because no more than 15 such clusters fit on the GPU at once.)
Plan plan_cosine(int M_tok, int N_out, int K, int sms) {
    const Plan ps = plan_slices(M_tok, N_out, K, sms);
    return make_plan(M_tok, N_out, K, ps.BN, 1, kSmemPair, false, 4 * kCosRed * 4);
}

template <class Epi>
cudaError_t launch_plan(const Plan &p, bool indep, const bf16 *W, int N_out, int K, const bf16 *X,
                        int M_tok, const Epi &epi, bool w_const, unsigned *status, cudaStream_t st,
                        unsigned *zero = nullptr, int nzero = 0) {
    if (p.stages < 2) return cudaErrorInvalidValue;
    CUtensorMap tmW, tmX;
    if (!make_tmap(&tmW, W, (uint64_t)N_out, (uint64_t)K, BM) ||
        !make_tmap(&tmX, X, (uint64_t)M_tok, (uint64_t)K, (uint32_t)p.xrows))
        return cudaErrorInvalidValue;
    // a weight matrix beyond 1/8 of L2 that one token tile reads once is streamed, not
    // reused: evict-first lines (with several token tiles its tiles are re-read)
    const int w_stream = p.tok_tiles == 1 && (size_t)N_out * (size_t)K * 2 > (size_t)16 << 20 ? 1 : 0;
    Shape g{M_tok, N_out, K, p.BN, p.splits, p.stages, w_const ? 1 : 0, indep ? 1 : 0, p.body,
            p.xrows, p.base_aligned, p.col_bytes, w_stream, zero, zero ? nzero : 0};
    // one CTA per SM (the shared memory of two exceeds an SM): 16 epilogue warps
    const bool wide = !Epi::kTileReduce && p.smem > (size_t)kSmemPair;
    auto kern = wide ? k_gemm_tc<Epi, 16> : k_gemm_tc<Epi, 8>;
    static bool configured[64] = {};   // per device: raise the shared-memory limit once (both kernels)
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(k_gemm_tc<Epi, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_gemm_tc<Epi, 16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = true;
    }
    return launch_kernel(kern, dim3(p.tok_tiles, p.w_tiles, p.splits), dim3(64 + 32 * (wide ? 16 : 8)), p.smem, st,
                         indep ? 1 : p.splits, tmW, tmX, g, epi, status);
}

}  // namespace

template <class Epi>
cudaError_t gemm_tc(const bf16 *W, int N_out, int K, const bf16 *X, int M_tok, const Epi &epi,
                    int splits, bool w_const, unsigned *status, cudaStream_t st) {
    if (M_tok <= 0 || N_out <= 0) return cudaSuccess;
    if (K % BK != 0 || N_out % 32 != 0) return cudaErrorInvalidValue;
    return launch_plan(plan_gemm(M_tok, N_out, K, splits, num_sms()), false, W, N_out, K, X, M_tok, epi,
                       w_const, status, st);
}

int gemm_tc_slices_count(int M_tok, int N_out, int K) {
    if (M_tok <= 0 || N_out <= 0 || K % BK != 0) return 1;
    return plan_slices(M_tok, N_out, K, num_sms()).splits;
}

int gemm_tc_plan_info(int M_tok, int N_out, int K, int splits_req, int sms, int kind, int *info) {
    if (M_tok <= 0 || N_out <= 0 || K <= 0 || K % BK != 0 || N_out % 32 != 0 || sms <= 0) return -1;
    if (kind == 2 && N_out > BM) return -1;
    const Plan p = kind == 1   ? plan_slices(M_tok, N_out, K, sms)
                   : kind == 2 ? plan_cosine(M_tok, N_out, K, sms)
                               : plan_gemm(M_tok, N_out, K, splits_req, sms);
    info[0] = p.BN;
    info[1] = p.splits;
    info[2] = p.stages;
    info[3] = p.tok_tiles;
    info[4] = p.w_tiles;
    info[5] = p.xrows;
    info[6] = (int)p.smem;
    info[7] = p.smem <= (size_t)kSmemPair ? 2 : 1;   // CTAs that fit on one SM
    return 0;
}

cudaError_t gemm_tc_slices(const bf16 *W, int N_out, int K, const bf16 *X, int M_tok, float *parts,
                           bool w_const, unsigned *status, cudaStream_t st, unsigned *zero, int nzero) {
    if (M_tok <= 0 || N_out <= 0) return cudaSuccess;
    if (K % BK != 0 || N_out % 32 != 0) return cudaErrorInvalidValue;
    const Plan p = plan_slices(M_tok, N_out, K, num_sms());
    EpiStoreF32 epi{SelRows{}, parts, N_out, N_out};
    return launch_plan(p, true, W, N_out, K, X, M_tok, epi, w_const, status, st, zero, nzero);
}

bool gemm_tc_cosine_ok(int M_tok, int N_out, int K) {
    return M_tok > 0 && N_out > 0 && N_out <= BM && N_out % 32 == 0 && K % BK == 0 &&
           plan_slices(M_tok, N_out, K, num_sms()).splits == 1;
}

cudaError_t gemm_tc_cosine(const bf16 *W, int N_out, int K, const bf16 *X, int M_tok, float *cur,
                           const float *cached, float *drift, bool w_const, unsigned *status, cudaStream_t st) {
    if (M_tok <= 0) return cudaSuccess;
    if (!gemm_tc_cosine_ok(M_tok, N_out, K)) return cudaErrorInvalidValue;
    const Plan p = plan_cosine(M_tok, N_out, K, num_sms());
    EpiCosine epi{SelRows{}, cur, cached, drift, N_out};
    return launch_plan(p, false, W, N_out, K, X, M_tok, epi, w_const, status, st);
}

template cudaError_t gemm_tc<EpiStoreF32>(const bf16 *, int, int, const bf16 *, int,
                                          const EpiStoreF32 &, int, bool, unsigned *, cudaStream_t);
template cudaError_t gemm_tc<EpiVocabStats>(const bf16 *, int, int, const bf16 *, int,
                                            const EpiVocabStats &, int, bool, unsigned *, cudaStream_t);
template cudaError_t gemm_tc<EpiQKV<bf16>>(const bf16 *, int, int, const bf16 *, int,
                                           const EpiQKV<bf16> &, int, bool, unsigned *, cudaStream_t);
template cudaError_t gemm_tc<EpiResidual<bf16>>(const bf16 *, int, int, const bf16 *, int,
                                                const EpiResidual<bf16> &, int, bool, unsigned *,
                                                cudaStream_t);
template cudaError_t gemm_tc<EpiSwiGLU<bf16>>(const bf16 *, int, int, const bf16 *, int,
                                              const EpiSwiGLU<bf16> &, int, bool, unsigned *,
                                              cudaStream_t);
template cudaError_t gemm_tc<EpiResidualNorm<bf16>>(const bf16 *, int, int, const bf16 *, int,
                                                    const EpiResidualNorm<bf16> &, int, bool, unsigned *,
                                                    cudaStream_t);
template cudaError_t gemm_tc<EpiSwiGLUNorm<bf16>>(const bf16 *, int, int, const bf16 *, int,
                                                  const EpiSwiGLUNorm<bf16> &, int, bool, unsigned *,
                                                  cudaStream_t);
template cudaError_t gemm_tc<EpiDownScatter<bf16>>(const bf16 *, int, int, const bf16 *, int,
                                                   const EpiDownScatter<bf16> &, int, bool, unsigned *,
                                                   cudaStream_t);

}  // namespace dllm
