// internal.h -- host-side interface between the C entry points (api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "epilogues.cuh"

namespace dllm {

int num_sms();   // SMs of the current device (cached per device)

bool pdl_enabled();   // programmatic dependent launch of the step's kernels (default on)

// Launches `kern` with the step's launch attributes: programmatic stream
// serialization (when enabled) and, for cluster_z > 1, a 1 x 1 x cluster_z cluster.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t st, int cluster_z, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (cluster_z > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = 1;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = cluster_z;
        ++n;
    }
    if (pdl_enabled()) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------- GEMMs
// acc[f, m] = <W[f, :K], X[m, :K]>, W [N_out, K] and X [M_tok, K] row-major,
// handed to `epi` (see epilogues.cuh).  N_out % 32 == 0.
//
// Tensor cores (bf16, tcgen05 + TMA): K % 64 == 0, rows 16-byte aligned.
// `splits` = 0 picks the K split (cluster size) automatically.
template <class Epi>
cudaError_t gemm_tc(const bf16 *W, int N_out, int K, const bf16 *X, int M_tok, const Epi &epi,
                    int splits, bool w_const, unsigned *status, cudaStream_t st);

// Independent K slices: parts[z * M_tok + m, f] = partial sum of slice z (fp32), for a
// later fixed-order reduction; gemm_tc_slices_count() tells how many slices it uses.
int gemm_tc_slices_count(int M_tok, int N_out, int K);
// The plan the tensor-core GEMM would launch for this shape on `sms` SMs, computed on the
// host only (no device query): info = {BN, splits, stages, token tiles, weight tiles,
// staged token rows, shared-memory bytes, CTAs per SM}.  kind 0: gemm_tc; 1: the
// independent-K-slice plan of gemm_tc_slices; 2: the plan of gemm_tc_cosine.  Returns -1
// for a shape the GEMM rejects.
int gemm_tc_plan_info(int M_tok, int N_out, int K, int splits_req, int sms, int kind, int *info);
// zero [nzero] (optional): words the first CTA clears after the previous kernel has
// completed, for the counters of the kernel that follows.
cudaError_t gemm_tc_slices(const bf16 *W, int N_out, int K, const bf16 *X, int M_tok, float *parts,
                           bool w_const, unsigned *status, cudaStream_t st, unsigned *zero = nullptr,
                           int nzero = 0);
// The singular proxy with its cosine drift in one launch (EpiCosine): cur [M_tok, N_out] =
// X W^T and drift [M_tok] against cached [M_tok, N_out]; needs N_out <= 128, N_out % 32 == 0,
// K % 64 == 0 and a shape whose slice plan has no K split (gemm_tc_cosine_ok).  No workspace.
bool gemm_tc_cosine_ok(int M_tok, int N_out, int K);
cudaError_t gemm_tc_cosine(const bf16 *W, int N_out, int K, const bf16 *X, int M_tok, float *cur,
                           const float *cached, float *drift, bool w_const, unsigned *status, cudaStream_t st);

// CUDA cores (fp32 FMA): any K.  zero [nzero] (optional) as for gemm_tc_slices.
template <class Epi>
cudaError_t gemm_simt(const float *W, int N_out, int K, const float *X, int M_tok, const Epi &epi,
                      cudaStream_t st, unsigned *zero = nullptr, int nzero = 0);

// ---------------------------------------------------------------- row kernels
template <class T>
cudaError_t gather_rmsnorm(const T *H, SelRows sel, int B, int d, const T *gamma, float eps, T *Xn,
                           float *proxy_cache, const float *proxy_cur, int r, const float *inv_freq,
                           int half_hd, float2 *rope_cs, unsigned *status, cudaStream_t st);

template <class T>
cudaError_t rmsnorm_rows(const float *h1, int M, int d, const T *gamma, float eps, T *Xn2,
                         cudaStream_t st);

// cur = sum of nparts partial proxies (parts[z * rows * r ...], fixed order; when
// nparts == 1, parts is cur itself), then drift = 1 - cos(cur, cached).  r <= 1024.
cudaError_t cosine_drift(const float *parts, int nparts, const float *cached, float *cur,
                         float *drift, long rows, int r, cudaStream_t st);

// Confidence extrapolation (ce.cu): one predict + update of every token's (level,
// velocity) Kalman state and the early-commit decision; M <= 1024 positions per sequence.
struct CEParams {
    float q_l, q_v, R, p_v0, z, c_min;
    int h_max;
};
cudaError_t ce_step(const float *conf, const uint8_t *seen, const uint8_t *undecided,
                    const uint8_t *committed, float *state, uint8_t *early, int B, int M,
                    const CEParams &p, cudaStream_t st);

// Drift-aware commit (polestar.cu): n = B * M tokens, history [n][2] (sum, count) fp32.
cudaError_t polestar_commit(const float *drift, const float *conf, const uint8_t *undecided,
                            const uint8_t *suffix, const uint8_t *selected, float *history, uint8_t *commit,
                            long n, float alpha, float tau_s, cudaStream_t st);

// Cluster-granular proxy (cluster.cu): spherical k-means over [B, N, D] rows with K
// centroids per sequence (C normalised first, `iters` Lloyd rounds, final assignment and
// row norms); residuals against the centroid direction; NVFP4 quantisation of [rows, D]
// (D % 16 == 0); selection of the kc most drifted clusters' rows (K <= 256).
cudaError_t spherical_kmeans(const float *X, float *C, int32_t *assign, float *xnorm, int B, int N, int D, int K,
                             int iters, cudaStream_t st);
cudaError_t cluster_residual(const float *X, const float *C, const int32_t *assign, const float *xnorm, float *R,
                             int B, int N, int D, int K, cudaStream_t st);
cudaError_t nvfp4_quantize(const float *R, float g, uint8_t *codes, uint8_t *scales, long rows, int D,
                           cudaStream_t st);
cudaError_t nvfp4_dequantize(const uint8_t *codes, const uint8_t *scales, float g, float *out, long rows, int D,
                             cudaStream_t st);
cudaError_t cluster_select(const float *Cn, const float *Cp, const int32_t *assign, int kc, int32_t *idx,
                           int32_t *count, int B, int N, int D, int K, cudaStream_t st);

// KL divergence of proxy-attention rows between two steps (kl.cu): drift [B, N] from
// cur, cache [B, N, r] fp32; r % 32 == 0, r <= 256.  Per-slice row states go to ws
// (kl_drift_workspace_bytes), merged by a second kernel.
int kl_drift_slices(int B, int N);
size_t kl_drift_workspace_bytes(int B, int N);
cudaError_t kl_drift(const float *cur, const float *cache, float *drift, int B, int N, int r, void *ws,
                     cudaStream_t st);

template <class T>
cudaError_t pack_rows_rope(const T *src, T *dst, int rows, int cols, int hd, cudaStream_t st);

template <class T>
cudaError_t pack_rows_interleave(const T *a, const T *b, T *dst, int rows, int cols,
                                 cudaStream_t st);

cudaError_t rope_inv_freq(float *dst, int hd, float theta, cudaStream_t st);

template <class T>
cudaError_t embed_rows(const T *E, const int32_t *tokens, const int32_t *rows, int R, T *H, int B,
                       int N, int d, int V, cudaStream_t st);

// dst[t][b * k_max + s] = src[t] row (b, idx[b, s]) of vecs[t] 16-byte units for the live
// rows, else 0; up to kGatherMax caches sharing one selection in one launch
// (dllm_gather_rows packs one, dllm_gather_rows_n several).
constexpr int kGatherMax = 4;
struct GatherSet {
    const void *src[kGatherMax];
    void *dst[kGatherMax];
    int vecs[kGatherMax];
};
cudaError_t gather_rows(const GatherSet &gs, int n, SelRows sel, int B, cudaStream_t st);

template <class T>
cudaError_t rows_rmsnorm(const T *H, const int32_t *rows, int R, const T *gamma, float eps, T *out,
                         int B, int N, int d, cudaStream_t st);

// One CTA waits on an mbarrier nothing completes (bounded wait); gave_up counts the
// threads whose wait ran out.
cudaError_t wait_timeout_check(int32_t *gave_up, unsigned *status, cudaStream_t st);

// ---------------------------------------------------------------- attention
// A[m, h*hd:(h+1)*hd] = softmax(Q_h K_g^T / sqrt(hd)) V_g over all N rows of the
// row's sequence, g = h / (n_q / n_kv); rows that are not live get zeros.
template <class T>
cudaError_t attention_simt(const T *Q, const T *Kc, const T *Vc, T *A, SelRows sel, int B,
                           int n_q, int n_kv, int hd, cudaStream_t st);

// Tensor cores (bf16, hd in {64, 128}); the key range is split over a cluster of up to
// 8 CTAs (attention_tc_splits) merged through distributed shared memory: no workspace.
int attention_tc_splits(int B, int k_max, int n_q, int N);

cudaError_t attention_tc(const bf16 *Q, const bf16 *Kc, const bf16 *Vc, bf16 *A, SelRows sel, int B,
                         int n_q, int n_kv, int hd, unsigned *status, cudaStream_t st);

// ---------------------------------------------------------------- selection
cudaError_t select_topk(const float *drift, const int32_t *forced, int F, int k, float min_drift,
                        int32_t *idx, int32_t *count, int B, int N, cudaStream_t st);

// Selection fused with the gather of the selected rows (front.cu): idx / count as
// select_topk, and for rows m = b * k_max + s the outputs of gather_rmsnorm.  N <= 4096.
// With dp.parts set, the kernel first computes drift [B, N] (and proxy_cur) from the
// proxy projection's K-slice partials, as cosine_drift would (r <= 128), its CTAs meeting
// at a per-sequence barrier on dp.arrive [B] (zero at launch); the grid must then fit on
// the GPU at once (select_gather_fused_ok).
struct DriftParts {
    const float *parts;   // [nparts, B*N, r] fp32 (nparts = 1: the proxies themselves, in
                          // proxy_cur), or nullptr: drift is an input
    int nparts;
    unsigned *arrive;     // [B] arrival counters, zeroed before the launch
};
int select_gather_max_n();
bool select_gather_fused_ok(int B, int N, int k_max, int dtype);
template <class T>
cudaError_t select_gather(float *drift, const int32_t *forced, int F, int k, float min_drift, int32_t *idx,
                          int32_t *count, int B, int N, int k_max, const T *H, int d, const T *gamma, float eps,
                          T *Xn, float *proxy_cache, float *proxy_cur, int r, const float *inv_freq,
                          int half_hd, float2 *rope_cs, DriftParts dp, unsigned *status, cudaStream_t st);

// ---------------------------------------------------------------- vocabulary
size_t commit_ws_bytes(int B, int M, int V);
// The commit step from per-slice states part[(b * M + m) * slices + i] (M <= 1024).
cudaError_t commit_from_states(const VocabState *part, int slices, const uint8_t *valid, int B, int M,
                               float conf_thresh, float tau, int32_t *token, float *conf, float *entropy,
                               float *max_entropy, int32_t *full_next, cudaStream_t st);
cudaError_t commit_entropy(const float *logits, const uint8_t *valid, int B, int M, int V,
                           float conf_thresh, float tau, int32_t *token, float *conf,
                           float *entropy, float *max_entropy, int32_t *full_next, void *ws,
                           cudaStream_t st);

}  // namespace dllm

namespace dllm {
// Allocation-free vocabulary step (scratch in a device array of the library).
int commit_noalloc_max_states();
size_t commit_noalloc_states(int B, int M, int V);
cudaError_t commit_entropy_noalloc(const float *logits, const uint8_t *valid, int B, int M, int V,
                                   float conf_thresh, float tau, int32_t *token, float *conf,
                                   float *entropy, float *max_entropy, int32_t *full_next,
                                   cudaStream_t st);
}  // namespace dllm
