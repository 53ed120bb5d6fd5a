// kl.cu -- drift of a row as the KL divergence between its attention distributions at two
// consecutive steps ("Polestar: drift-aware cache correction and token commit", 2. A,
// Polestar-Cache, drift measurement: D_i = KL(A_i^t || A_i^{t-1})), over row-granular proxy
// attention: A_i(j) = softmax_j(<s_i, s_j> / sqrt(r)) over the other rows j != i of the
// sequence, with the singular proxies of this step (A^t) and the cached ones (A^{t-1}).  The
// row's own column is left out: with the same proxy as query and key its logit |s_i|^2 /
// sqrt(r) would dominate and every distribution would be one-hot on itself.
//
// With x_j = <cur_i, cur_j> / sqrt(r), y_j = <cache_i, cache_j> / sqrt(r), p = softmax(x):
//     D_i = sum_j p_j (x_j - y_j) - (LSE(x) - LSE(y)),   LSE(x) = m_x + ln sum_j e^(x_j - m_x),
// and D_i = 0 for a sequence of one row.
// One pass over the keys keeps, per row, the running maxima m_x, m_y, the sums
// Z_x = sum e^(x - m_x), Z_y = sum e^(y - m_y) and W = sum e^(x - m_x) (x - y), rescaled
// whenever a maximum grows.  Identical proxies give x == y bit for bit, hence W = 0,
// Z_x == Z_y and D = 0 exactly.
//
// fp32 on the CUDA cores: the drift is made of score differences that bf16 tensor-core
// scores would swamp.  One CTA (8 warps) = 64 query rows x one slice of the 128-row key
// tiles; thread (ty, tx) owns rows 8 ty .. 8 ty + 7 and key columns 4 tx .. 4 tx + 3 of both
// score tiles (64 FMA per 6 shared-memory loads, issued as 32 packed two-lane FMAs on
// row pairs), so one warp holds eight whole rows of a
// tile.  The query tile (both steps, all
// r dimensions) stays in shared memory, transposed; the key tiles stream through a two-chunk
// ring of 32 dimensions each, the next chunk's global loads held in registers while the
// current chunk is multiplied.  The shared memory (~134 KB at r = 128) keeps one CTA per SM,
// and the number of key slices is chosen so that every CTA runs in one wave.  Each slice
// writes its per-row (m_x, Z_x, W, m_y, Z_y) to the workspace; a second kernel merges the
// slices of every row in slice order.  (Merging inside a thread-block cluster instead left
// some 8-CTA clusters for a second wave.)
#include <math.h>

#include "internal.h"

namespace dllm {
namespace {

constexpr int kQ = 64;           // query rows per CTA
constexpr int kK = 128;          // key rows per tile
constexpr int kR = 32;           // proxy dimensions per staged chunk
constexpr int kPq = kQ + 4;      // padded rows of the transposed chunks (16-byte aligned)
constexpr int kPk = kK + 4;
constexpr int kThreads = 256;    // 8 x 32 threads, 8 x 4 scores each
constexpr int kWarps = kThreads / 32;
constexpr int kRows = kQ / kWarps;   // query rows per thread (and per warp)
constexpr int kMaxSlices = 32;
constexpr int kMaxR = 256;

// dynamic shared memory: query tile [2 steps][r][kPq], key ring [2 buffers][2 steps][kR][kPk]
__host__ __device__ inline size_t kl_smem_bytes(int r) {
    return ((size_t)2 * r * kPq + (size_t)4 * kR * kPk) * 4;
}

struct RowState {
    float mx, zx, w, my, zy;
};

// Chunk [row0, row0 + ROWS) x [c0, c0 + 32) of a [N, r] matrix as ROWS / kWarps values per
// thread (dimension = lane, rows warp + kWarps i; rows past N are zero), and its transposed
// store dst[c * P + row].
template <int ROWS>
__device__ __forceinline__ void load_chunk(float (&v)[ROWS / kWarps], const float *__restrict__ src, int row0,
                                           int N, int r, int c0) {
    const int c = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int i = 0; i < ROWS / kWarps; ++i) {
        const int row = row0 + w + kWarps * i;
        v[i] = row < N ? src[(size_t)row * r + c0 + c] : 0.f;
    }
}
template <int ROWS, int P>
__device__ __forceinline__ void store_chunk(float *dst, const float (&v)[ROWS / kWarps]) {
    const int c = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int i = 0; i < ROWS / kWarps; ++i) dst[c * P + w + kWarps * i] = v[i];
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__global__ void __launch_bounds__(kThreads, 1)
    k_kl_slices(const float *__restrict__ cur, const float *__restrict__ cache, RowState *__restrict__ part,
                int B, int N, int r, int S) {
    extern __shared__ __align__(16) float smf[];
    float *qc = smf;                    // [r][kPq] this step's query proxies, transposed
    float *qp = qc + (size_t)r * kPq;   // [r][kPq] the cached ones
    float *ring = qp + (size_t)r * kPq; // [2 buffers][2 steps][kR][kPk]

    griddep_wait();
    griddep_launch();
    const int b = blockIdx.y;
    const int q0 = blockIdx.x * kQ;
    const int slice = (int)blockIdx.z;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const float *cb = cur + (size_t)b * N * r;
    const float *pb = cache + (size_t)b * N * r;
    const float scale = 1.f / sqrtf((float)r);

    const int nkt = (N + kK - 1) / kK;
    const int kt0 = (int)((long long)slice * nkt / S), kt1 = (int)((long long)(slice + 1) * nkt / S);
    const int nch = r / kR;
    const int nit = (kt1 - kt0) * nch;

    // the query tile (four chunks' loads in flight before they are stored) and the first key chunk
    for (int c0 = 0; c0 < r; c0 += 4 * kR) {
        float v[4][kQ / kWarps];
        const int n = (r - c0) / kR < 4 ? (r - c0) / kR : 4;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (k < n) load_chunk<kQ>(v[k], cb, q0, N, r, c0 + k * kR);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (k < n) store_chunk<kQ, kPq>(qc + (size_t)(c0 + k * kR) * kPq, v[k]);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (k < n) load_chunk<kQ>(v[k], pb, q0, N, r, c0 + k * kR);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (k < n) store_chunk<kQ, kPq>(qp + (size_t)(c0 + k * kR) * kPq, v[k]);
    }
    float pc_[kK / kWarps], pp_[kK / kWarps];
    if (nit > 0) {
        load_chunk<kK>(pc_, cb, kt0 * kK, N, r, 0);
        load_chunk<kK>(pp_, pb, kt0 * kK, N, r, 0);
        store_chunk<kK, kPk>(ring, pc_);
        store_chunk<kK, kPk>(ring + kR * kPk, pp_);
    }
    __syncthreads();

    float mx[kRows], zx[kRows], w[kRows], my[kRows], zy[kRows];
#pragma unroll
    for (int a = 0; a < kRows; ++a) {
        mx[a] = -INFINITY;
        my[a] = -INFINITY;
        zx[a] = 0.f;
        zy[a] = 0.f;
        w[a] = 0.f;
    }
    // score accumulators of row pairs (2h, 2h+1) x column e: one packed fp32 FMA updates
    // both rows (each lane of the pair rounds exactly as a scalar fmaf would)
    float2 xx[kRows / 2][4], yy[kRows / 2][4];
    for (int it = 0; it < nit; ++it) {
        const int kt = kt0 + it / nch, ch = it % nch;
        const int k0 = kt * kK;
        if (ch == 0) {
#pragma unroll
            for (int h = 0; h < kRows / 2; ++h)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    xx[h][e] = make_float2(0.f, 0.f);
                    yy[h][e] = make_float2(0.f, 0.f);
                }
        }
        if (it + 1 < nit) {   // next chunk's loads in flight during this chunk's products
            const int nk0 = (kt0 + (it + 1) / nch) * kK, nc0 = ((it + 1) % nch) * kR;
            load_chunk<kK>(pc_, cb, nk0, N, r, nc0);
            load_chunk<kK>(pp_, pb, nk0, N, r, nc0);
        }
        const float *kcb = ring + (size_t)(it & 1) * 2 * kR * kPk;
        const float *kpb = kcb + kR * kPk;
        const float *qcb = qc + (size_t)ch * kR * kPq;
        const float *qpb = qp + (size_t)ch * kR * kPq;
#pragma unroll 8
        for (int c = 0; c < kR; ++c) {
            const float4 ac0 = *reinterpret_cast<const float4 *>(qcb + c * kPq + ty * kRows);
            const float4 ac1 = *reinterpret_cast<const float4 *>(qcb + c * kPq + ty * kRows + 4);
            const float4 ap0 = *reinterpret_cast<const float4 *>(qpb + c * kPq + ty * kRows);
            const float4 ap1 = *reinterpret_cast<const float4 *>(qpb + c * kPq + ty * kRows + 4);
            const float4 bc = *reinterpret_cast<const float4 *>(kcb + c * kPk + tx * 4);
            const float4 bp = *reinterpret_cast<const float4 *>(kpb + c * kPk + tx * 4);
            const float2 av[kRows / 2] = {make_float2(ac0.x, ac0.y), make_float2(ac0.z, ac0.w),
                                          make_float2(ac1.x, ac1.y), make_float2(ac1.z, ac1.w)};
            const float2 pv[kRows / 2] = {make_float2(ap0.x, ap0.y), make_float2(ap0.z, ap0.w),
                                          make_float2(ap1.x, ap1.y), make_float2(ap1.z, ap1.w)};
            const float bv[4] = {bc.x, bc.y, bc.z, bc.w}, qv[4] = {bp.x, bp.y, bp.z, bp.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 be = make_float2(bv[e], bv[e]), qe = make_float2(qv[e], qv[e]);
#pragma unroll
                for (int h = 0; h < kRows / 2; ++h) {
                    xx[h][e] = __ffma2_rn(av[h], be, xx[h][e]);
                    yy[h][e] = __ffma2_rn(pv[h], qe, yy[h][e]);
                }
            }
        }
        if (it + 1 < nit) {   // the other buffer was last read in iteration it - 1
            float *nb = ring + (size_t)((it + 1) & 1) * 2 * kR * kPk;
            store_chunk<kK, kPk>(nb, pc_);
            store_chunk<kK, kPk>(nb + kR * kPk, pp_);
        }
        __syncthreads();
        if (ch != nch - 1) continue;
        float x[kRows][4], y[kRows][4];
#pragma unroll
        for (int h = 0; h < kRows / 2; ++h)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                x[2 * h][e] = xx[h][e].x;
                x[2 * h + 1][e] = xx[h][e].y;
                y[2 * h][e] = yy[h][e].x;
                y[2 * h + 1][e] = yy[h][e].y;
            }
        // online update of the thread's rows over this tile's live key columns (j < N, j != i)
#pragma unroll
        for (int a = 0; a < kRows; ++a) {
            const int qi = q0 + ty * kRows + a;
            float tmx = -INFINITY, tmy = -INFINITY;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                x[a][e] *= scale;
                y[a][e] *= scale;
                const int j = k0 + tx * 4 + e;
                if (j < N && j != qi) {
                    tmx = fmaxf(tmx, x[a][e]);
                    tmy = fmaxf(tmy, y[a][e]);
                }
            }
            tmx = warp_max(tmx);   // -inf only if the tile's one live key is the row itself
            tmy = warp_max(tmy);
            const float nmx = fmaxf(mx[a], tmx), nmy = fmaxf(my[a], tmy);
            float sx = 0.f, sw = 0.f, sy = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = k0 + tx * 4 + e;
                if (j < N && j != qi) {
                    const float ex = expf(x[a][e] - nmx);
                    sx += ex;
                    sw = fmaf(ex, x[a][e] - y[a][e], sw);
                    sy += expf(y[a][e] - nmy);
                }
            }
            sx = warp_sum(sx);
            sw = warp_sum(sw);
            sy = warp_sum(sy);
            // rescale of the running sums: 0 when they were empty, 1 when the maximum held
            // (also while no live key has been seen, where both maxima are still -inf)
            const float cx = mx[a] == nmx ? 1.f : expf(mx[a] - nmx);
            const float cy = my[a] == nmy ? 1.f : expf(my[a] - nmy);
            zx[a] = fmaf(zx[a], cx, sx);
            w[a] = fmaf(w[a], cx, sw);
            zy[a] = fmaf(zy[a], cy, sy);
            mx[a] = nmx;
            my[a] = nmy;
        }
    }
    if (tx == 0)
#pragma unroll
        for (int a = 0; a < kRows; ++a) {
            const int qi = q0 + ty * kRows + a;
            if (qi < N) part[((size_t)slice * B + b) * N + qi] = RowState{mx[a], zx[a], w[a], my[a], zy[a]};
        }
}

// D of every row from its S slice states, merged in slice order.
__global__ void __launch_bounds__(256)
    k_kl_merge(const RowState *__restrict__ part, float *__restrict__ drift, long rows, int S) {
    griddep_wait();
    griddep_launch();
    const long t = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= rows) return;
    float Mx = -INFINITY, My = -INFINITY;
    for (int s = 0; s < S; ++s) {
        const RowState p = part[(size_t)s * rows + t];
        if (p.zx > 0.f) {
            Mx = fmaxf(Mx, p.mx);
            My = fmaxf(My, p.my);
        }
    }
    float Zx = 0.f, W = 0.f, Zy = 0.f;
    for (int s = 0; s < S; ++s) {
        const RowState p = part[(size_t)s * rows + t];
        if (!(p.zx > 0.f)) continue;   // a slice without keys for this row
        const float cx = expf(p.mx - Mx), cy = expf(p.my - My);
        Zx = fmaf(p.zx, cx, Zx);
        W = fmaf(p.w, cx, W);
        Zy = fmaf(p.zy, cy, Zy);
    }
    drift[t] = Zx > 0.f ? W / Zx - (Mx - My) - (logf(Zx) - logf(Zy)) : 0.f;
}

}  // namespace

// Key slices per query tile: as many as keep every CTA (one per SM) in one wave.
int kl_drift_slices(int B, int N) {
    const int nqt = (N + kQ - 1) / kQ, nkt = (N + kK - 1) / kK;
    const long long tiles = (long long)nqt * B;
    int s = (int)(num_sms() / tiles);
    s = s < 1 ? 1 : (s > kMaxSlices ? kMaxSlices : s);
    return s > nkt ? nkt : s;
}

size_t kl_drift_workspace_bytes(int B, int N) {
    if (B <= 0 || N <= 0) return 0;
    return (size_t)kl_drift_slices(B, N) * B * N * sizeof(RowState) + 256;
}

cudaError_t kl_drift(const float *cur, const float *cache, float *drift, int B, int N, int r, void *ws,
                     cudaStream_t st) {
    if (B <= 0 || N <= 0) return cudaSuccess;
    if (r <= 0 || r % kR != 0 || r > kMaxR || B > 65535 || !ws) return cudaErrorInvalidValue;
    static bool configured[64] = {};   // per device: raise the dynamic shared-memory limit once
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !configured[dev]) {
        const cudaError_t e = cudaFuncSetAttribute(k_kl_slices, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)kl_smem_bytes(kMaxR));
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) configured[dev] = true;
    }
    const int S = kl_drift_slices(B, N);
    RowState *part = reinterpret_cast<RowState *>((reinterpret_cast<uintptr_t>(ws) + 255) & ~uintptr_t(255));
    const dim3 grid((unsigned)((N + kQ - 1) / kQ), (unsigned)B, (unsigned)S);
    cudaError_t e = launch_kernel(k_kl_slices, grid, dim3(kThreads), kl_smem_bytes(r), st, 1, cur, cache, part,
                                  B, N, r, S);
    if (e != cudaSuccess) return e;
    const long rows = (long)B * N;
    return launch_kernel(k_kl_merge, dim3((unsigned)((rows + 255) / 256)), dim3(256), 0, st, 1,
                         (const RowState *)part, drift, rows, S);
}

}  // namespace dllm
