// attention_tc.cu -- non-causal attention of the selected queries over the whole
// partially refreshed cache on the sm_103a tensor cores (SPA-Cache, "3. Sparse
// execution": the sparse queries attend to the partially updated KV cache).
//
// One CTA = 128 selected rows of one sequence (MMA M) x one query head x one
// slice of the key range.  Per 128-key tile:
//   S  = Q K^T          tcgen05.mma, Q and K K-major (head dim contiguous), fp32 in TMEM
//   P  = exp2(S*c - m)  softmax warps, bf16 into shared memory in the 128-byte-swizzled
//                       K-major layout
//   PV = P V            tcgen05.mma, V read MN-major (head dim contiguous), fp32 in TMEM
//   O  = O * corr + PV  in registers (streaming softmax)
// K and V tiles are double-buffered by TMA; S is double-buffered in TMEM so the next
// tile's Q K^T runs while the softmax of the current one is computed.  Keys beyond N
// are masked.  With several key slices, the slices of one (rows, head) tile run as a
// thread-block cluster: each keeps its (O, m, l) in shared memory and the CTAs merge
// disjoint row ranges through distributed shared memory (no workspace, no second launch).
//
// Roles (64 + 128 SG threads): warp 0 TMA, warp 1 TMEM owner + MMA issuer, the other warps
// softmax: SG warps per TMEM lane quarter, thread = (query row, 1/SG of the key and head
// columns).  The kernel takes the whole SM (one CTA).  With few key tiles per CTA (the
// batch-1 steps) a tile's dependent chain sets the time and SG = 4 shortens it; with many
// (long contexts, batches) SG = 2 exchanges less per tile and keeps the pipe busier.
#include <cudaTypedefs.h>

#include "internal.h"

namespace dllm {

bool make_tmap(CUtensorMap *tm, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows);

namespace {

constexpr int AQ = 128;          // query rows per CTA
constexpr int AKV = 128;         // keys per tile

constexpr int kChunk = 128 * 128;   // one 64-column (128-byte) box of 128 rows: 16 KB

struct AttnArgs {
    const int32_t *count;
    int N, k_max, n_q, n_kv, B;
    int kv_tiles, splits, q_tiles;
    float scale_log2;                 // log2(e) / sqrt(hd)
    bf16 *A;                          // [B*k_max, n_q*hd]
};

// 2^x by the SFU's approximate base-2 exponential (relative error ~2^-22, subnormal
// results flushed to zero; 2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <int HD, int SG>
__global__ void __launch_bounds__(64 + 128 * SG, 1)
    k_attention_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const AttnArgs a, unsigned *status) {
    constexpr int NCH = HD / 64;               // 64-column boxes per row of Q / K / V
    constexpr int QB = NCH * kChunk;           // bytes of the Q tile
    constexpr int KB = NCH * kChunk;           // bytes of one K (or V) tile
    constexpr int PB = 2 * kChunk;             // P tile: 128 rows x 128 keys bf16
    constexpr int kSoftThreads = 128 * SG;
    constexpr int OH = HD / SG;                // head-dim columns per thread
    constexpr int KC = AKV / SG;               // key columns per thread and tile
    extern __shared__ uint8_t smem_raw[];
    const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    uint8_t *smem = smem_raw + pad;
    uint8_t *sQ = smem;
    uint8_t *sK = sQ + QB;                     // [2][KB]
    uint8_t *sV = sK + 2 * KB;                 // [2][KB]
    uint8_t *sP = sV + 2 * KB;                 // [PB]
    float *xmax = reinterpret_cast<float *>(sP + PB);   // [SG][128] exchange between a row's threads
    float *xsum = xmax + 128 * SG;                       // [SG][128]
    uint64_t *bars = reinterpret_cast<uint64_t *>(xsum + 128 * SG);
    uint64_t *q_full = bars + 0;
    uint64_t *k_full = bars + 1;               // [2]
    uint64_t *v_full = bars + 3;               // [2]
    uint64_t *k_empty = bars + 5;              // [2] K tile read by its S product
    uint64_t *s_full = bars + 7;               // [2]
    uint64_t *s_free = bars + 9;               // [2]
    uint64_t *p_full = bars + 11;
    uint64_t *pv_full = bars + 12;
    uint64_t *v_empty = bars + 13;             // [2] V tile read by its PV product
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 15);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q0 = blockIdx.x * AQ;
    const int h = blockIdx.y;
    const int b = blockIdx.z / a.splits;
    const int split = blockIdx.z - b * a.splits;
    const int g = h / (a.n_q / a.n_kv);
    const int t0 = (int)((long long)split * a.kv_tiles / a.splits);
    const int t1 = (int)((long long)(split + 1) * a.kv_tiles / a.splits);
    const int nt = t1 - t0;
    const int dq = a.n_q * HD;
    const size_t row0 = (size_t)b * a.k_max + q0;   // flattened row of query 0

    // barriers, descriptors and tensor memory first: none of it reads what the previous
    // kernel writes, so it overlaps that kernel's tail
    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_empty[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&s_free[i], kSoftThreads);
        }
        mbar_init(p_full, kSoftThreads);
        mbar_init(pv_full, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS[2] = {tmem, tmem + 128};
    const uint32_t tPV = tmem + 256;

    griddep_wait();
    griddep_launch();
    int live = a.count[b];
    live = live < a.k_max ? live : a.k_max;
    live -= q0;                                 // live query rows of this tile
    if (live <= 0) {   // no live query (the same in every slice of the cluster): zero outputs
        if (split == 0 && warp >= 2) {
            const int r = (warp & 3) * 32 + lane, qt = (warp - 2) >> 2;
            if (q0 + r < a.k_max) {
                bf16 *dst = a.A + (row0 + r) * dq + (size_t)h * HD + qt * OH;
                for (int e = 0; e < OH; ++e) dst[e] = __float2bfloat16_rn(0.f);
            }
        }
        tc_fence_before();
        __syncthreads();
        if (warp == 1) {
            tc_fence_after();
            tmem_dealloc(tmem, 512);
        }
        return;
    }

    // softmax threads' results for the key-split merge: (O row half, m, l) of the row
    float o[OH];
    float m_fin = -INFINITY, l_fin = 0.f;
    if (warp == 0) {
        // ---------------- TMA producers: lane 0 loads Q and the K tiles, lane 1 the V tiles;
        // a K buffer is refilled as soon as its Q K^T product is done, a V buffer after
        // its P V product
        if (lane == 0) {
            mbar_arrive_expect_tx(q_full, QB);
            for (int c = 0; c < NCH; ++c)
                tma_load_2d(sQ + c * kChunk, &tmQ, q_full, h * HD + c * 64, (int)row0);
        }
        if (lane < 2) {
            const bool isK = lane == 0;
            uint64_t *fullb = isK ? k_full : v_full;
            uint64_t *emptyb = isK ? k_empty : v_empty;
            uint8_t *buf = isK ? sK : sV;
            const CUtensorMap *tm = isK ? &tmK : &tmV;
            int issued = 0;
            for (int it = 0; it < nt; ++it) {
                const int s = it & 1;
                const uint32_t ph = (uint32_t)(it >> 1) & 1u;
                if (!mbar_wait(&emptyb[s], ph ^ 1u, abort_flag, status)) break;
                const int y = b * a.N + (t0 + it) * AKV;
                mbar_arrive_expect_tx(&fullb[s], KB);
                for (int c = 0; c < NCH; ++c)
                    tma_load_2d(buf + s * KB + c * kChunk, tm, &fullb[s], g * HD + c * 64, y);
                ++issued;
            }
            if (*abort_flag) {   // every issued copy must land before the CTA can exit
                if (isK) mbar_drain(q_full, 0);
                for (int it = issued > 2 ? issued - 2 : 0; it < issued; ++it)
                    mbar_drain(&fullb[it & 1], (uint32_t)(it >> 1) & 1u);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {   // ---------------- MMA issuer
            const uint32_t id_s = idesc_bf16(128, AKV, 0);
            const uint32_t id_pv = idesc_bf16(128, HD, 1);
            const uint32_t aq = smem_u32(sQ), ak = smem_u32(sK), av = smem_u32(sV), ap = smem_u32(sP);
            bool ok = mbar_wait(q_full, 0, abort_flag, status);
            auto issue_s = [&](int it) -> bool {
                const int s = it & 1;
                const uint32_t ph = (uint32_t)(it >> 1) & 1u;
                if (!mbar_wait(&s_free[s], ph ^ 1u, abort_flag, status)) return false;
                if (!mbar_wait(&k_full[s], ph, abort_flag, status)) return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk) {
                    const uint32_t off = (uint32_t)((kk >> 2) * kChunk + (kk & 3) * 32);
                    mma_bf16(tS[s], smem_desc_sw128(aq + off, 16, 1024),
                             smem_desc_sw128(ak + s * KB + off, 16, 1024), id_s, kk > 0);
                }
                mma_commit(&s_full[s]);
                mma_commit(&k_empty[s]);   // the K buffer may be refilled
                return true;
            };
            if (ok && nt > 0) ok = issue_s(0);
            for (int it = 0; ok && it < nt; ++it) {
                if (it + 1 < nt && !issue_s(it + 1)) break;
                const int s = it & 1;
                const uint32_t ph = (uint32_t)(it >> 1) & 1u;
                if (!mbar_wait(p_full, (uint32_t)it & 1u, abort_flag, status)) break;
                if (!mbar_wait(&v_full[s], ph, abort_flag, status)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < AKV / 16; ++kk) {
                    // P: K-major, keys 16kk.. (+32 B inside the swizzled row, 16 KB per 64 keys)
                    const uint32_t offp = (uint32_t)((kk >> 2) * kChunk + (kk & 3) * 32);
                    // V: MN-major, keys 16kk.. start 16 rows (2 KB) further; LBO = next 64 dims
                    const uint32_t offv = (uint32_t)(kk * 16 * 128);
                    mma_bf16(tPV, smem_desc_sw128(ap + offp, 16, 1024),
                             smem_desc_sw128(av + s * KB + offv, kChunk, 1024), id_pv, kk > 0);
                }
                mma_commit(pv_full);
                mma_commit(&v_empty[s]);
            }
        }
    } else {   // ---------------- softmax warps: thread = (query row, quarter)
        const int q = warp & 3;
        const int qt = (warp - 2) >> 2;              // key columns qt*KC.., head dims qt*OH..
        const int r = q * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
#pragma unroll
        for (int e = 0; e < OH; ++e) o[e] = 0.f;
        float m_run = -INFINITY, l_run = 0.f;
        float corr_prev = 1.f;   // rescale factor of the PV product still in flight
        // P row r, keys qt*KC..: 64-key chunk qt*KC / 64, first 16-byte unit (qt*KC % 64) / 8
        uint8_t *prow = sP + (qt * KC / 64) * kChunk + (r >> 3) * 1024 + (r & 7) * 128;
        const int u0 = (qt * KC % 64) / 8;
        // O <- O * corr + PV of the previous tile (its MMA overlapped this tile's softmax)
        auto fold_pv = [&](int tile) -> bool {
            if (!mbar_wait(pv_full, (uint32_t)tile & 1u, abort_flag, status)) return false;
            tc_fence_after();
#pragma unroll
            for (int c0 = 0; c0 < OH; c0 += 16) {
                float t[16];
                tmem_ld_x16(tPV + lane_addr + (uint32_t)(qt * OH + c0), t);
                tmem_ld_wait(t);
#pragma unroll
                for (int j = 0; j < 16; ++j) o[c0 + j] = fmaf(o[c0 + j], corr_prev, t[j]);
            }
            return true;
        };
        bool ok = true;
        for (int it = 0; it < nt && ok; ++it) {
            const int s = it & 1;
            const uint32_t ph = (uint32_t)(it >> 1) & 1u;
            if (!mbar_wait(&s_full[s], ph, abort_flag, status)) { ok = false; break; }
            tc_fence_after();
            const int nvalid = a.N - (t0 + it) * AKV - qt * KC;   // keys of my quarter inside [0, N)
            float v[KC];
#pragma unroll
            for (int c0 = 0; c0 < KC; c0 += 16)
                tmem_ld_x16(tS[s] + lane_addr + (uint32_t)(qt * KC + c0), slice16(v + c0));
#pragma unroll
            for (int c0 = 0; c0 < KC; c0 += 16) tmem_ld_wait(slice16(v + c0));
            tc_fence_before();
            mbar_arrive(&s_free[s]);                    // S buffer may be overwritten now
            if (nvalid < KC) {   // keys past N (last tile only): out of the max and the sum
#pragma unroll
                for (int j = 0; j < KC; ++j)
                    if (j >= nvalid) v[j] = -INFINITY;
            }
            float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int j = 0; j < KC; ++j) mq[j & 3] = fmaxf(mq[j & 3], v[j]);
            float mt = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
            xmax[qt * 128 + r] = mt;
            named_bar_sync(2 + q, 32 * SG);            // the SG warps of this lane quarter
#pragma unroll
            for (int p = 0; p < SG; ++p) mt = fmaxf(mt, xmax[p * 128 + r]);
            const float m_new = fmaxf(m_run, mt * a.scale_log2);
            const float corr = ex2_approx(m_run - m_new);
            float ls[4] = {0.f, 0.f, 0.f, 0.f};
            uint32_t pk[KC / 2];                       // P of this tile, bf16 pairs
#pragma unroll
            for (int j = 0; j < KC; j += 2) {          // 2^(-inf) = 0 for the masked keys
                const float p0 = ex2_approx(fmaf(v[j], a.scale_log2, -m_new));
                const float p1 = ex2_approx(fmaf(v[j + 1], a.scale_log2, -m_new));
                const __nv_bfloat162 pp = __floats2bfloat162_rn(p0, p1);
                ls[(j >> 1) & 3] += __low2float(pp) + __high2float(pp);
                pk[j >> 1] = *reinterpret_cast<const uint32_t *>(&pp);
            }
            const float lsum = (ls[0] + ls[1]) + (ls[2] + ls[3]);
            // the P buffer is free once the previous tile's PV product has completed
            if (it > 0 && !(ok = fold_pv(it - 1))) break;
#pragma unroll
            for (int c0 = 0; c0 < KC; c0 += 8) {
                const int u = (u0 + (c0 >> 3)) ^ (r & 7);   // 16-byte unit in the swizzled row
                *reinterpret_cast<uint4 *>(prow + u * 16) =
                    make_uint4(pk[c0 / 2], pk[c0 / 2 + 1], pk[c0 / 2 + 2], pk[c0 / 2 + 3]);
            }
            fence_proxy_async_smem();
            mbar_arrive(p_full);
            l_run = l_run * corr + lsum;
            m_run = m_new;
            corr_prev = corr;
        }
        if (ok && nt > 0) fold_pv(nt - 1);
        // combine the row's quarter sums (the same order in every thread of the row)
        xsum[qt * 128 + r] = l_run;
        named_bar_sync(2 + q, 32 * SG);
        float l_tot = 0.f;
#pragma unroll
        for (int p = 0; p < SG; ++p) l_tot += xsum[p * 128 + r];
        const bool row_ok = q0 + r < a.k_max;
        const size_t row = row0 + r;
        m_fin = (r < live && nt > 0) ? m_run : -INFINITY;
        l_fin = (r < live && nt > 0) ? l_tot : 0.f;
        if (a.splits == 1) {
            if (row_ok) {
                const float inv = (r < live && l_tot > 0.f) ? 1.0f / l_tot : 0.f;
                bf16 *dst = a.A + row * dq + (size_t)h * HD + qt * OH;
                // 16-byte stores (8 dims): the 32 lanes of a warp write 32 different rows
#pragma unroll
                for (int e = 0; e < OH; e += 8) {
                    uint4 u;
                    const __nv_bfloat162 p0 = __floats2bfloat162_rn(o[e] * inv, o[e + 1] * inv);
                    const __nv_bfloat162 p1 = __floats2bfloat162_rn(o[e + 2] * inv, o[e + 3] * inv);
                    const __nv_bfloat162 p2 = __floats2bfloat162_rn(o[e + 4] * inv, o[e + 5] * inv);
                    const __nv_bfloat162 p3 = __floats2bfloat162_rn(o[e + 6] * inv, o[e + 7] * inv);
                    u.x = *reinterpret_cast<const uint32_t *>(&p0);
                    u.y = *reinterpret_cast<const uint32_t *>(&p1);
                    u.z = *reinterpret_cast<const uint32_t *>(&p2);
                    u.w = *reinterpret_cast<const uint32_t *>(&p3);
                    *reinterpret_cast<uint4 *>(dst + e) = u;
                }
            }
        }
    }
    __syncwarp();
    if (a.splits > 1) {
        // The key slices of one (rows, head) tile are the CTAs of a cluster; CTA rank k
        // owns rows [k*per, (k+1)*per).  Once every CTA is past its main loop (first
        // barrier), each pushes its (O, m, l) of every row into the owner's shared memory
        // (remote stores, over the owner's idle Q tile and K ring); after the second
        // barrier every owner merges its rows from local memory.
        const int S = a.splits;
        const int per = (AQ + S - 1) / S;
        const uint32_t my = cluster_ctarank();
        float *rO = reinterpret_cast<float *>(smem);   // [S senders][per rows][HD]
        float *rML = rO + (size_t)S * per * HD;         // [S senders][per rows][m, l]
        cluster_sync_all();
        if (warp >= 2) {
            const int q = warp & 3, qt = (warp - 2) >> 2, r = q * 32 + lane;
            const int owner = r / per, lr = r - owner * per;
            const uint32_t dO = mapa_shared(smem_u32(rO + ((size_t)(my * per + lr) * HD + qt * OH)), (uint32_t)owner);
#pragma unroll
            for (int e = 0; e < OH; e += 4)
                st_dsmem_f32x4(dO + (uint32_t)(e * 4), make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]));
            if (qt == 0) {
                const uint32_t dM = mapa_shared(smem_u32(rML + (size_t)(my * per + lr) * 2), (uint32_t)owner);
                st_dsmem_f32(dM, m_fin);
                st_dsmem_f32(dM + 4, l_fin);
            }
        }
        __syncwarp();
        cluster_sync_all();   // every push has landed; nothing remote is touched after this
        if (warp >= 2) {
            const int tid = threadIdx.x - 64;
            const int rb = (int)my * per;
            const int nrows = min(per, AQ - rb);
            constexpr int D4 = HD / 4;
            for (int it = tid; it < nrows * D4; it += kSoftThreads) {
                const int lr = it / D4, d4 = it - lr * D4;
                float M = -INFINITY;
                for (int sp = 0; sp < S; ++sp) M = fmaxf(M, rML[(sp * per + lr) * 2]);
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                float den = 0.f;
                if (M != -INFINITY) {
                    for (int sp = 0; sp < S; ++sp) {
                        const float ms = rML[(sp * per + lr) * 2];
                        if (ms == -INFINITY) continue;
                        const float w = ex2_approx(ms - M);
                        den = fmaf(rML[(sp * per + lr) * 2 + 1], w, den);
                        const float4 x = *reinterpret_cast<const float4 *>(rO + ((size_t)(sp * per + lr) * HD + d4 * 4));
                        acc.x = fmaf(x.x, w, acc.x);
                        acc.y = fmaf(x.y, w, acc.y);
                        acc.z = fmaf(x.z, w, acc.z);
                        acc.w = fmaf(x.w, w, acc.w);
                    }
                }
                const int rr = rb + lr;
                if (q0 + rr < a.k_max) {
                    const float iv = den > 0.f ? 1.0f / den : 0.f;
                    __nv_bfloat162 *dst = reinterpret_cast<__nv_bfloat162 *>(
                        a.A + (row0 + rr) * dq + (size_t)h * HD + d4 * 4);
                    const __nv_bfloat162 p0 = __floats2bfloat162_rn(acc.x * iv, acc.y * iv);
                    const __nv_bfloat162 p1 = __floats2bfloat162_rn(acc.z * iv, acc.w * iv);
                    uint2 u;   // one 8-byte store
                    u.x = *reinterpret_cast<const uint32_t *>(&p0);
                    u.y = *reinterpret_cast<const uint32_t *>(&p1);
                    *reinterpret_cast<uint2 *>(dst) = u;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int HD, int SG>
size_t attn_smem() {
    return 1024 + (size_t)(HD / 64) * kChunk * 5 + 2 * kChunk + 2 * 128 * SG * 4 + 16 * 8 + 64;
}

}  // namespace

int attention_tc_splits(int B, int k_max, int n_q, int N) {
    const int qt = (k_max + AQ - 1) / AQ;
    const long long base = (long long)qt * n_q * B;
    const int kv_tiles = (N + AKV - 1) / AKV;
    // one CTA per SM (the ring and TMEM need the whole SM): as many key slices as keep
    // the grid within a single wave; the slices of a tile form a cluster (at most 8)
    int s = (int)(num_sms() / base);
    if (s > kv_tiles) s = kv_tiles;
    if (s > 8) s = 8;
    return s < 1 ? 1 : s;
}

cudaError_t attention_tc(const bf16 *Q, const bf16 *Kc, const bf16 *Vc, bf16 *A, SelRows sel, int B,
                         int n_q, int n_kv, int hd, unsigned *status, cudaStream_t st) {
    const int M = B * sel.k_max;
    if (M <= 0) return cudaSuccess;
    if (hd != 64 && hd != 128) return cudaErrorInvalidValue;
    CUtensorMap tq, tk, tv;
    const int dq = n_q * hd, dkv = n_kv * hd;
    if (!make_tmap(&tq, Q, (uint64_t)M, (uint64_t)dq, AQ) ||
        !make_tmap(&tk, Kc, (uint64_t)B * sel.N, (uint64_t)dkv, AKV) ||
        !make_tmap(&tv, Vc, (uint64_t)B * sel.N, (uint64_t)dkv, AKV))
        return cudaErrorInvalidValue;
    AttnArgs a{};
    a.count = sel.count;
    a.N = sel.N;
    a.k_max = sel.k_max;
    a.n_q = n_q;
    a.n_kv = n_kv;
    a.B = B;
    a.kv_tiles = (sel.N + AKV - 1) / AKV;
    a.splits = attention_tc_splits(B, sel.k_max, n_q, sel.N);
    a.q_tiles = (sel.k_max + AQ - 1) / AQ;
    a.scale_log2 = 1.4426950408889634f / sqrtf((float)hd);
    a.A = A;
    dim3 grid(a.q_tiles, n_q, B * a.splits);
    // threads per query row: 4 when each CTA runs few key tiles (latency), else 2
    const int tiles_per_cta = (a.kv_tiles + a.splits - 1) / a.splits;
    const bool sg4 = tiles_per_cta <= 8;
    static bool configured[64] = {};   // per device: raise the shared-memory limit once
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        cudaError_t e = cudaFuncSetAttribute(k_attention_tc<128, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)attn_smem<128, 2>());
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_attention_tc<128, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)attn_smem<128, 4>());
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_attention_tc<64, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)attn_smem<64, 2>());
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_attention_tc<64, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)attn_smem<64, 4>());
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = true;
    }
    if (hd == 128)
        return sg4 ? launch_kernel(k_attention_tc<128, 4>, grid, dim3(64 + 128 * 4), attn_smem<128, 4>(), st, a.splits, tq,
                                   tk, tv, a, status)
                   : launch_kernel(k_attention_tc<128, 2>, grid, dim3(64 + 128 * 2), attn_smem<128, 2>(), st, a.splits, tq,
                                   tk, tv, a, status);
    return sg4 ? launch_kernel(k_attention_tc<64, 4>, grid, dim3(64 + 128 * 4), attn_smem<64, 4>(), st, a.splits, tq, tk,
                               tv, a, status)
               : launch_kernel(k_attention_tc<64, 2>, grid, dim3(64 + 128 * 2), attn_smem<64, 2>(), st, a.splits, tq, tk,
                               tv, a, status);
}

}  // namespace dllm
