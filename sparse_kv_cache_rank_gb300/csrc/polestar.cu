// polestar.cu -- drift-aware token commit ("Polestar: drift-aware cache correction and token
// commit", 2. B, Polestar-Commit).  A current-block token commits when its drift delta (its
// drift minus the mean of its earlier drifts) exceeds the confidence-conditioned threshold
// alpha (tau_s - c)^2; a suffix token commits when the drift score selected it at this step
// and its confidence reaches tau_s.  Every token's drift history (sum, count) then takes this
// step's drift.  Elementwise over the B x M tokens.
#include "internal.h"

namespace dllm {
namespace {

__global__ void __launch_bounds__(256)
    k_polestar_commit(const float *__restrict__ drift, const float *__restrict__ conf,
                      const uint8_t *__restrict__ undecided, const uint8_t *__restrict__ suffix,
                      const uint8_t *__restrict__ selected, float2 *__restrict__ hist,
                      uint8_t *__restrict__ commit, long n, float alpha, float tau_s) {
    griddep_wait();
    griddep_launch();
    const long t = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= n) return;
    const float d = drift[t], c = conf[t];
    const float2 h = hist[t];   // (sum of earlier drifts, their count)
    uint8_t go = 0;
    if (undecided[t]) {
        if (suffix[t]) {
            go = selected[t] != 0 && c >= tau_s;
        } else if (h.y >= 1.f) {
            const float delta = d - h.x / h.y;
            const float g = tau_s - c;
            go = delta > alpha * g * g;
        }
    }
    commit[t] = go;
    hist[t] = make_float2(h.x + d, h.y + 1.f);
}

}  // namespace

cudaError_t polestar_commit(const float *drift, const float *conf, const uint8_t *undecided,
                            const uint8_t *suffix, const uint8_t *selected, float *history, uint8_t *commit,
                            long n, float alpha, float tau_s, cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    const unsigned blocks = (unsigned)((n + 255) / 256);
    return launch_kernel(k_polestar_commit, dim3(blocks), dim3(256), 0, st, 1, drift, conf, undecided, suffix,
                         selected, reinterpret_cast<float2 *>(history), commit, n, alpha, tau_s);
}

}  // namespace dllm
