// select.cu -- per-sequence top-k of the drift scores (SPA-Cache, "1. Update
// identification via singular proxy" and "2. Adaptive budget allocation") united
// with the always-recomputed rows (EntropyCache, "How EntropyCache works", step 3).
//
// One CTA per sequence (256 threads up to N = 4096, 1024 above), keys in shared memory.  The k-th largest
// drift is found exactly by a 4-pass radix select on order-preserving 32-bit keys
// (256-bin shared histograms); rows above it are taken, rows equal to it are taken
// in index order until the budget is met (lower row index wins ties), and the union
// with the forced rows is compacted in ascending order by a block-wide scan.
#include "select.cuh"

namespace dllm {
namespace {

constexpr int kTMax = 1024;
constexpr int kMaxN = 16384;

template <int kT>
__global__ void __launch_bounds__(kT) k_select_topk(const float *__restrict__ drift,
                                                    const int32_t *__restrict__ forced, int F, int k,
                                                    float min_drift, int32_t *__restrict__ idx,
                                                    int32_t *__restrict__ count, int N) {
    extern __shared__ uint32_t sm[];
    uint32_t *key = sm;                                          // [N] 0 = not eligible
    uint8_t *flag = reinterpret_cast<uint8_t *>(key + N);        // [N] 1 = forced
    griddep_wait();
    griddep_launch();
    const int b = blockIdx.x;
    const uint32_t total = select_sequence<kT>(drift + (size_t)b * N, forced ? forced + (size_t)b * F : nullptr, F, k,
                                               min_drift, N, key, flag, idx + (size_t)b * N);
    if (threadIdx.x == 0) count[b] = (int32_t)total;
}

}  // namespace

cudaError_t select_topk(const float *drift, const int32_t *forced, int F, int k, float min_drift,
                        int32_t *idx, int32_t *count, int B, int N, cudaStream_t st) {
    if (B <= 0 || N <= 0) return cudaSuccess;
    if (N > kMaxN) return cudaErrorInvalidValue;
    const size_t smem = (size_t)N * 5;
    // fewer threads (cheaper block barriers) while each still handles <= 16 rows
    if (N <= 4096) {
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(k_select_topk<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
        }
        return launch_kernel(k_select_topk<256>, dim3(B), dim3(256), smem, st, 1, drift, forced, F, k,
                             min_drift, idx, count, N);
    }
    cudaError_t e = cudaFuncSetAttribute(k_select_topk<kTMax>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_kernel(k_select_topk<kTMax>, dim3(B), dim3(kTMax), smem, st, 1, drift, forced, F, k,
                         min_drift, idx, count, N);
}

}  // namespace dllm

// ---------------------------------------------------------------------------
// Diagnostic of the bounded wait (dllm_check_wait_timeout): every thread waits on a
// barrier whose phase never completes; each wait must give up after the limit and
// return false, and the status word must receive DLLM_STATUS_TIMEOUT.
namespace dllm {
namespace {

__global__ void __launch_bounds__(64) k_wait_timeout(int32_t *gave_up, unsigned *status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const bool ok = mbar_wait(&bar, 0, &abort, status);
    if (!ok) atomicAdd(gave_up, 1);
}

}  // namespace

cudaError_t wait_timeout_check(int32_t *gave_up, unsigned *status, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(gave_up, 0, sizeof(int32_t), st);
    if (e != cudaSuccess) return e;
    return launch_kernel(k_wait_timeout, dim3(1), dim3(64), 0, st, 1, gave_up, status);
}

}  // namespace dllm
