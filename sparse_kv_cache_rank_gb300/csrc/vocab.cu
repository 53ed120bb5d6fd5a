// vocab.cu -- the vocabulary-side decision (EntropyCache, "How EntropyCache works",
// steps 2-3; TSPD "Input features"; Polestar "1. Problem definition").
//
// Pass 1 streams each logit row once (one CTA per row slice) and keeps, per thread,
// the running state of the row's softmax in a single sweep:
//   m = max logit, a = its lowest index, s = sum e^(l - m), t = sum (l - m) e^(l - m),
// so that p_max = 1/s and entropy = -sum p ln p = ln s - t/s.  States merge exactly
// under a change of reference maximum m -> M:  s' = s e^(m-M), t' = e^(m-M)(t + (m-M) s).
// Pass 2 (one CTA per sequence) merges the slices of each row and applies the commit
// rule and the full-refresh decision.
#include <cfloat>
#include <mutex>

#include "internal.h"

namespace dllm {
namespace {

using RowState = VocabState;

__device__ __forceinline__ RowState merge(RowState x, RowState y) { return vocab_merge(x, y); }

constexpr int kT1 = 256;

__global__ void __launch_bounds__(kT1) k_row_stats(const float *__restrict__ logits,
                                                   const uint8_t *__restrict__ valid, int V,
                                                   int slices, RowState *__restrict__ part) {
    griddep_wait();
    griddep_launch();
    const int row = blockIdx.y, sl = blockIdx.x;
    if (!valid[row]) return;
    const int chunk = (V + slices - 1) / slices;
    const int v0 = sl * chunk, v1 = min(V, v0 + chunk);
    const float *l = logits + (size_t)row * V;
    RowState st{-INFINITY, 0.f, 0.f, INT_MAX};
    for (int v = v0 + threadIdx.x; v < v1; v += kT1) {
        const float x = l[v];
        if (st.s == 0.f) {
            st = RowState{x, 1.f, 0.f, v};
        } else if (x > st.m) {
            const float c = expf(st.m - x);
            st.t = c * (st.t + (st.m - x) * st.s);
            st.s = st.s * c + 1.f;
            st.m = x;
            st.a = v;
        } else {
            const float e = expf(x - st.m);
            st.s += e;
            st.t = fmaf(x - st.m, e, st.t);
        }
    }
    // warp then block merge
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        RowState y;
        y.m = __shfl_xor_sync(0xffffffffu, st.m, o);
        y.s = __shfl_xor_sync(0xffffffffu, st.s, o);
        y.t = __shfl_xor_sync(0xffffffffu, st.t, o);
        y.a = __shfl_xor_sync(0xffffffffu, st.a, o);
        st = merge(st, y);
    }
    __shared__ RowState ws[kT1 / 32];
    if ((threadIdx.x & 31) == 0) ws[threadIdx.x >> 5] = st;
    __syncthreads();
    if (threadIdx.x == 0) {
        RowState r = ws[0];
        for (int w = 1; w < kT1 / 32; ++w) r = merge(r, ws[w]);
        part[(size_t)row * slices + sl] = r;
    }
}

// One CTA per sequence, thread m = row m of the block of candidates.
__global__ void __launch_bounds__(1024) k_commit(const RowState *__restrict__ part, int slices,
                                                 const uint8_t *__restrict__ valid, int M,
                                                 float conf_thresh, float tau, int32_t *token,
                                                 float *conf, float *entropy, float *max_entropy,
                                                 int32_t *full_next) {
    griddep_wait();
    griddep_launch();
    const int b = blockIdx.x, m = threadIdx.x;
    __shared__ float s_conf[32];
    __shared__ int s_row[32];
    __shared__ unsigned s_emax;
    __shared__ RowState s_state[1024];
    if (m == 0) s_emax = 0u;
    // each row's slices merged by one warp: lane-strided in slice order, then a butterfly
    // (a fixed order, so results repeat exactly)
    {
        const int warp = m >> 5, lane = m & 31, nwarps = blockDim.x >> 5;
        for (int row = warp; row < M; row += nwarps) {
            RowState r{-INFINITY, 0.f, 0.f, INT_MAX};
            if (valid[(size_t)b * M + row]) {
                const RowState *ps = part + ((size_t)b * M + row) * slices;
                for (int i = lane; i < slices; i += 32) r = merge(r, ps[i]);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    RowState y;
                    y.m = __shfl_xor_sync(0xffffffffu, r.m, o);
                    y.s = __shfl_xor_sync(0xffffffffu, r.s, o);
                    y.t = __shfl_xor_sync(0xffffffffu, r.t, o);
                    y.a = __shfl_xor_sync(0xffffffffu, r.a, o);
                    r = (lane & o) ? merge(y, r) : merge(r, y);
                }
            }
            if (lane == 0) s_state[row] = r;
        }
    }
    __syncthreads();
    const bool live = m < M && valid[(size_t)b * M + m];
    float p = 0.f, H = 0.f;
    int am = -1;
    if (live) {
        const RowState r = s_state[m];
        p = 1.0f / r.s;
        H = fmaxf(logf(r.s) - r.t / r.s, 0.f);
        am = r.a;
    }
    if (m < M) {
        conf[(size_t)b * M + m] = p;
        entropy[(size_t)b * M + m] = H;
    }
    const bool pass = live && p >= conf_thresh;
    const int any = __syncthreads_or(pass);
    // highest confidence among live rows, lowest row on ties (used when none passes)
    float bc = live ? p : -1.f;
    int br = live ? m : INT_MAX;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float oc = __shfl_xor_sync(0xffffffffu, bc, o);
        const int orow = __shfl_xor_sync(0xffffffffu, br, o);
        if (oc > bc || (oc == bc && orow < br)) {
            bc = oc;
            br = orow;
        }
    }
    if ((m & 31) == 0) {
        s_conf[m >> 5] = bc;
        s_row[m >> 5] = br;
    }
    __syncthreads();
    if (m < 32) {
        const int nw = (blockDim.x + 31) / 32;
        bc = m < nw ? s_conf[m] : -1.f;
        br = m < nw ? s_row[m] : INT_MAX;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float oc = __shfl_xor_sync(0xffffffffu, bc, o);
            const int orow = __shfl_xor_sync(0xffffffffu, br, o);
            if (oc > bc || (oc == bc && orow < br)) {
                bc = oc;
                br = orow;
            }
        }
        if (m == 0) s_row[0] = bc >= 0.f ? br : -1;
    }
    __syncthreads();
    const bool commit = any ? pass : (live && m == s_row[0]);
    if (m < M) token[(size_t)b * M + m] = commit ? am : -1;
    if (commit) atomicMax(&s_emax, __float_as_uint(H));   // H >= 0: bit order = value order
    __syncthreads();
    if (m == 0) {
        const float E = __uint_as_float(s_emax);
        max_entropy[b] = E;
        full_next[b] = E > tau ? 1 : 0;
    }
}

int slices_for(int rows, int V) {
    const int sms = num_sms();
    int s = (2 * sms + rows - 1) / (rows > 0 ? rows : 1);
    const int cap = (V + 2047) / 2048;
    if (s > cap) s = cap;
    return s < 1 ? 1 : s;
}

}  // namespace

size_t commit_ws_bytes(int B, int M, int V) {
    const int rows = B * M;
    return (size_t)rows * slices_for(rows, V) * sizeof(RowState);
}

cudaError_t commit_from_states(const VocabState *part, int slices, const uint8_t *valid, int B, int M,
                               float conf_thresh, float tau, int32_t *token, float *conf, float *entropy,
                               float *max_entropy, int32_t *full_next, cudaStream_t st) {
    if (B <= 0 || M <= 0) return cudaSuccess;
    // enough warps that each merges few rows (M <= 1024 threads for the per-row step)
    int threads = ((M + 31) / 32) * 32;
    const int want = 32 * (slices < 32 ? slices : 32);
    if (threads < want) threads = want;
    if (threads > 1024) threads = 1024;
    return launch_kernel(k_commit, dim3(B), dim3(threads), 0, st, 1, part, slices, valid, M, conf_thresh, tau,
                         token, conf, entropy, max_entropy, full_next);
}

cudaError_t commit_entropy(const float *logits, const uint8_t *valid, int B, int M, int V,
                           float conf_thresh, float tau, int32_t *token, float *conf,
                           float *entropy, float *max_entropy, int32_t *full_next, void *ws,
                           cudaStream_t st) {
    if (B <= 0) return cudaSuccess;
    const int rows = B * M;
    RowState *part = reinterpret_cast<RowState *>(ws);
    if (rows > 0) {
        const int slices = slices_for(rows, V);
        cudaError_t e = launch_kernel(k_row_stats, dim3(slices, rows), dim3(kT1), 0, st, 1, logits, valid, V, slices, part);
        if (e != cudaSuccess) return e;
        return commit_from_states(part, slices, valid, B, M, conf_thresh, tau, token, conf, entropy,
                                  max_entropy, full_next, st);
    } else {
        const int threads = 32;
        return launch_kernel(k_commit, dim3(B), dim3(threads), 0, st, 1, part, 1, valid, 0, conf_thresh, tau, token, conf, entropy,
                                        max_entropy, full_next);
    }
    return cudaGetLastError();
}

}  // namespace dllm

// ---------------------------------------------------------------------------
// Allocation-free variant of the vocabulary step, for callers that cannot allocate
// device memory (no cudaMalloc and no caching allocator on their side, e.g. code that
// only ever receives buffers from a host application).  Its scratch (one softmax state
// per row slice) lives in this file-scope device array instead of a caller workspace;
// every GPU that loads the library keeps the array until the process exits.
namespace dllm {
namespace {

constexpr int kNoAllocStates = 16384;   // 16384 row-slice states x 16 bytes = 256 KB
__device__ __align__(256) RowState g_commit_scratch[kNoAllocStates];

// Device address of the scratch array on the current device (resolved once per device).
cudaError_t noalloc_scratch(RowState **out) {
    static RowState *addr[64] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_commit_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = static_cast<RowState *>(p);
    }
    *out = addr[dev];
    return cudaSuccess;
}

}  // namespace

int commit_noalloc_max_states() { return kNoAllocStates; }

size_t commit_noalloc_states(int B, int M, int V) {
    const int rows = B * M;
    return (size_t)rows * slices_for(rows, V);
}

cudaError_t commit_entropy_noalloc(const float *logits, const uint8_t *valid, int B, int M, int V,
                                   float conf_thresh, float tau, int32_t *token, float *conf,
                                   float *entropy, float *max_entropy, int32_t *full_next,
                                   cudaStream_t st) {
    RowState *scratch = nullptr;
    cudaError_t e = noalloc_scratch(&scratch);
    if (e != cudaSuccess) return e;
    // every state the commit kernel reads is written by the row kernel of this call,
    // so nothing has to be cleared between calls
    return commit_entropy(logits, valid, B, M, V, conf_thresh, tau, token, conf, entropy, max_entropy,
                          full_next, scratch, st);
}

}  // namespace dllm
