/*
 * dllm.h -- C ABI of the GB300 sparse KV-cache refresh library (libdllm.so).
 *
 * One denoising step of a bidirectional (non-causal) diffusion-LLM layer with a
 * sparse cache refresh, as stated by:
 *   [SPA] "Singular proxies for adaptive caching in diffusion language models"
 *         (SPA-Cache): "1. Update identification via singular proxy",
 *         "2. Adaptive budget allocation", "3. Sparse execution";
 *   [EC]  "EntropyCache": "How EntropyCache works", steps 1-3;
 *   [TSPD] "Efficient diffusion LLMs via temporal-spatial parallel decoding and
 *         confidence extrapolation": "Input features";
 *   [POL] "Polestar: drift-aware cache correction and token commit for efficient
 *         diffusion LLM inference": "1. Problem definition".
 *
 * Conventions shared by every call
 * --------------------------------
 * Memory    All array pointers are DEVICE pointers owned by the caller, C-contiguous,
 *           row-major with leading dimension equal to the logical width, and 16-byte
 *           aligned.  The library never allocates device memory: scratch space is
 *           the caller's workspace `ws` of `ws_bytes` bytes, sized by the matching
 *           *_workspace_bytes() query (256-byte aligned).  Outputs never alias inputs
 *           unless a parameter says so.
 * Streams   `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *           stream).  Every compute call only enqueues work and returns; nothing
 *           synchronises the host except dllm_check_status().
 * dtype     DLLM_BF16: hidden states, weights, K/V caches and gains are bf16 and every
 *           GEMM runs on the tcgen05 tensor cores with fp32 accumulation.
 *           DLLM_F32: the same arrays are fp32 and every product runs on the CUDA
 *           cores in fp32.  Proxies, drift, logits and all statistics are fp32 in
 *           both cases.
 * Errors    Every call returns DLLM_OK (0) or a negative code; the message of the
 *           last failure on the calling thread is dllm_last_error().  Argument errors
 *           are detected on the host before any launch.  Device-side conditions
 *           (a bounded wait that ran out, a count larger than k_max) set bits of a
 *           device status word read by dllm_check_status(); no kernel traps.
 */
#ifndef DLLM_H_
#define DLLM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DLLM_OK 0
#define DLLM_ERR_INVALID_ARG (-1) /* null pointer, bad size, misalignment, k > N ...  */
#define DLLM_ERR_UNSUPPORTED (-2) /* shape/dtype combination without a kernel          */
#define DLLM_ERR_WORKSPACE (-3)   /* ws_bytes smaller than the query returned          */
#define DLLM_ERR_CUDA (-4)        /* a CUDA runtime call or launch failed              */
#define DLLM_ERR_TIMEOUT (-5)     /* reported by dllm_check_status()                   */

#define DLLM_F32 0
#define DLLM_BF16 1

/* Device status bits (dllm_check_status). */
#define DLLM_STATUS_TIMEOUT 1u     /* a kernel's bounded mbarrier wait ran out          */
#define DLLM_STATUS_COUNT_CLAMP 2u /* count[b] > k_max: extra rows were ignored         */
#define DLLM_STATUS_SMEM_LAYOUT 4u /* a GEMM found its shared memory misaligned and      */
                                   /* skipped its work (outputs not written)             */

/* Message of the last failed call on this thread ("" if none). */
const char *dllm_last_error(void);

/* Library ABI version (major * 100 + minor): 1.00 holds the path's calls and the
 * allocation-free vocabulary step (dllm_commit_entropy_noalloc); 1.10 adds the NEXT-row
 * calls (KL drift, drift-aware commit, confidence extrapolation, cluster-granular
 * proxy); 1.11 the host-only GEMM plan query (dllm_gemm_plan); 1.12 the read-back of
 * refreshed rows (dllm_gather_rows), the bounded-wait diagnostic
 * (dllm_check_wait_timeout) and the one-call layer step (dllm_layer_step); 1.13 the
 * read-back of several caches' refreshed rows in one launch (dllm_gather_rows_n). */
int dllm_version(void);

/* Reads (and with reset != 0 clears) the device status word of the current device.
 * Synchronises the device.  Returns DLLM_ERR_TIMEOUT if the timeout bit is set,
 * DLLM_ERR_CUDA if the shared-memory layout bit is set, DLLM_OK otherwise;
 * *status_out (optional) receives all bits. */
int dllm_check_status(unsigned *status_out, int reset);

/* Diagnostic of the failure path that replaces traps (no counterpart on the pages): one
 * CTA of 64 threads waits, with the same bounded mbarrier wait every pipelined kernel of
 * the library uses, on a barrier that nothing ever completes.  The wait gives up after
 * its limit (1 s), raises DLLM_STATUS_TIMEOUT and the kernel returns; *gave_up (device,
 * int32) receives the number of threads whose wait returned false (64 when the path
 * works).  A following dllm_check_status() reports DLLM_ERR_TIMEOUT, and the context
 * stays usable.  Errors: INVALID_ARG (null gave_up), CUDA (launch). */
int dllm_check_wait_timeout(int32_t *gave_up, void *stream);

/* ---------------------------------------------------------------------------
 * [SPA] "1. Update identification via singular proxy"
 *
 * proxy_cur[t] = H[t] . P                 (t = b*N + i, P = Pt^T, [d x r])
 * drift[t]     = 1 - <proxy_cur[t], proxy_cache[t]> / sqrt(|proxy_cur[t]|^2 |proxy_cache[t]|^2)
 * with drift = 0 when both proxies are zero, 1 when exactly one is, and clamped to
 * [0, 2].  Identical proxies give exactly 0.
 *   H           [B, N, d]  dtype      layer input (residual stream before the norm)
 *   Pt          [r, d]     dtype      proxy matrix, transposed: row j = column j of
 *                                     U_r S_r of diag(gamma1) W_V^T (built once per layer)
 *   proxy_cache [B, N, r]  fp32       proxies stored when each row was last refreshed
 *   proxy_cur   [B, N, r]  fp32 out
 *   drift       [B, N]     fp32 out
 * Requirements: r % 32 == 0, r <= 1024; d % 64 == 0 for DLLM_BF16; B * N <= INT_MAX.
 * Workspace: dllm_proxy_workspace_bytes() bytes (fp32 partial proxies of independent K
 * slices, summed in a fixed order by a second kernel that computes the drift), 0 when
 * the shape needs no K split.  Without a split (bf16, r <= 128, the token tiles alone fill
 * the GPU) one launch computes the proxies and, in its epilogue, their drift.  Either way
 * identical inputs always give identical results.
 * ------------------------------------------------------------------------- */
size_t dllm_proxy_workspace_bytes(int B, int N, int d, int r, int dtype);

int dllm_proxy_score(const void *H, const void *Pt, const float *proxy_cache, float *proxy_cur,
                     float *drift, int B, int N, int d, int r, int dtype, void *ws,
                     size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * [POL] "2. A. Polestar-Cache", drift measurement: the drift of a row between
 * consecutive steps is the KL divergence of its attention distributions,
 * D_i = KL(A_i^t || A_i^{t-1}) -- an alternative score to the cosine of
 * dllm_proxy_score, selected on in the same way (dllm_select_topk).  The page gives
 * no formula for A; the attention here is row-granular proxy attention over the
 * other rows of the sequence:
 *   A^t_i(j)     = softmax over j != i of <proxy_cur[b,i], proxy_cur[b,j]> / sqrt(r)
 *   A^{t-1}_i(j) = the same with proxy_cache
 *   drift[b, i]  = sum_{j != i} A^t_i(j) ln(A^t_i(j) / A^{t-1}_i(j));  0 when N == 1.
 * Identical proxies give exactly 0.  fp32 arithmetic (CUDA cores).
 *   proxy_cur, proxy_cache [B, N, r] fp32 (as produced and kept by dllm_proxy_score);
 *   drift [B, N] fp32 out.
 * Workspace: dllm_kl_drift_workspace_bytes(B, N) bytes (per-row states of the key slices,
 * merged in a fixed order, so identical inputs always give identical results).
 * Requirements: r % 32 == 0, r <= 256, B <= 65535.  Caller-owned arrays; errors:
 * DLLM_ERR_ARG for null pointers or non-positive sizes, DLLM_ERR_UNSUPPORTED for r,
 * DLLM_ERR_WORKSPACE for a missing or short workspace.
 * ------------------------------------------------------------------------- */
size_t dllm_kl_drift_workspace_bytes(int B, int N);

int dllm_kl_drift(const float *proxy_cur, const float *proxy_cache, float *drift, int B, int N,
                  int r, void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * [TSPD] "2. Confidence Extrapolation (CE)": the top-1 confidence of every token is a
 * noisy observation of a latent (level, velocity) state, filtered like a Kalman filter;
 * near-future confidence is forecast with its uncertainty and a token is committed early
 * when a conservative lower bound of the forecast exceeds a minimum threshold, within a
 * look-ahead horizon bounded by the left context already fixed.  The page gives no
 * equations or constants; this call takes the textbook constant-velocity filter:
 *   seen[b,m] != 0:  predict l- = l + v, P- = F P F^T + diag(q_l, q_v) (F = [[1,1],[0,1]]),
 *                    update with c = conf[b,m]: S = P-00 + R, K = (P-00, P-10)/S,
 *                    l = l- + K0 (c - l-), v = v + K1 (c - l-), P = (I - K [1 0]) P-;
 *   seen[b,m] == 0:  l = c, v = 0, P = diag(R, p_v0) (first observation);
 *   H = min(h_max, #{m' < m : committed[b,m'] != 0});
 *   early[b,m] = undecided[b,m] && exists h in 1..H with
 *                l + h v - z sqrt(P00 + 2h P01 + h^2 P11) >= c_min.
 *   conf [B, M] fp32 (dllm_commit_entropy's conf); seen, undecided, committed [B, M] uint8;
 *   state [B, M, 5] fp32 (l, v, P00, P01, P11), read when seen and written for every
 *   position; early [B, M] uint8 out.
 * Requirements: M <= 1024, R > 0, noise levels >= 0, 0 <= h_max <= 1024.  No workspace.
 * ------------------------------------------------------------------------- */
int dllm_ce_step(const float *conf, const uint8_t *seen, const uint8_t *undecided,
                 const uint8_t *committed, float *state, uint8_t *early, int B, int M, float q_l,
                 float q_v, float R, float p_v0, float z, int h_max, float c_min, void *stream);

/* ---------------------------------------------------------------------------
 * [POL] "2. B. Polestar-Commit": a token of the current block is committed when its drift
 * delta (its drift minus the historical mean of its drift) exceeds the confidence-
 * conditioned threshold alpha (tau_s - c)^2; suffix tokens are committed when the drift
 * score selects them and their confidence reaches tau_s.  The page gives no alpha, tau_s or
 * history; this call takes the mean of the token's earlier drifts:
 *   current block (suffix == 0): commit = undecided && count >= 1 &&
 *                                 drift - sum / count > alpha (tau_s - conf)^2
 *   suffix (suffix != 0):        commit = undecided && selected && conf >= tau_s
 *   then history = (sum + drift, count + 1) for every token.
 *   drift, conf [B, M] fp32 (the step's drift score and top-1 confidence);
 *   undecided, suffix, selected [B, M] uint8; history [B, M, 2] fp32 (sum, count; zero to
 *   start), 8-byte aligned, updated in place; commit [B, M] uint8 out.
 * No workspace.
 * ------------------------------------------------------------------------- */
int dllm_polestar_commit(const float *drift, const float *conf, const uint8_t *undecided,
                         const uint8_t *suffix, const uint8_t *selected, float *history, uint8_t *commit,
                         int B, int M, float alpha, float tau_s, void *stream);

/* ---------------------------------------------------------------------------
 * [POL] "2. A. Polestar-Cache", local window and clustering / sparse updates: the hidden
 * states of a local window are clustered with spherical k-means, their residuals are
 * quantised with NVFP4 into a compressed proxy, and the top-k drifted clusters are
 * refreshed.  The page names the steps, not their equations; these calls take:
 *
 * dllm_spherical_kmeans: X [B, N, D] fp32 rows; C [B, K, D] fp32 initial centroids,
 *   normalised to unit length, then `iters` Lloyd rounds (a_i = argmax_k <x_i, c_k>, the
 *   lowest k on ties; c_k = normalise(sum of x_i / |x_i| over its members, in row order),
 *   an empty cluster keeps its centroid) and a final assignment; assign [B, N] int32 and
 *   xnorm [B, N] fp32 (|x_i|) out.  D % 4 == 0, D <= 8192, K <= 256, X and C
 *   16-byte aligned.
 * dllm_cluster_residual: R [B, N, D] = x_i - xnorm_i c_{assign_i} (an assignment outside
 *   [0, K) leaves the row whole).
 * dllm_nvfp4_quantize: R [rows, D] fp32 (16-byte aligned, D % 16 == 0), tensor scale g > 0;
 *   per 16-element block scales [rows, D/16] = E4M3(amax / (6 g)) and codes [rows, D/2]
 *   (8-byte aligned) = E2M1(x / (scale g)), two per byte, element 2j in the low nibble
 *   (sign << 3 | magnitude index into {0, .5, 1, 1.5, 2, 3, 4, 6}); both rounded to
 *   nearest even with saturation by the device conversions; code 0 when the scale is 0.
 * dllm_nvfp4_dequantize: out [rows, D] fp32 (16-byte aligned) = E2M1(code) * E4M3(scale) * g,
 *   the first product exact, one rounding by the multiplication with g.
 * dllm_cluster_select: drift_k = 1 - cos(C_now[b,k], C_prev[b,k]) (0 for two zero rows, 1
 *   for one); the kc clusters with the largest drift (lower k on ties); idx [B, N] receives
 *   their member rows ascending, then -1; count [B] their number (the same output as
 *   dllm_select_topk, for dllm_sparse_layer_refresh).  K <= 256.
 * No workspace.
 * ------------------------------------------------------------------------- */
int dllm_spherical_kmeans(const float *X, float *C, int32_t *assign, float *xnorm, int B, int N, int D, int K,
                          int iters, void *stream);
int dllm_cluster_residual(const float *X, const float *C, const int32_t *assign, const float *xnorm, float *R,
                          int B, int N, int D, int K, void *stream);
int dllm_nvfp4_quantize(const float *R, float g, uint8_t *codes, uint8_t *scales, long rows, int D, void *stream);
int dllm_nvfp4_dequantize(const uint8_t *codes, const uint8_t *scales, float g, float *out, long rows, int D,
                          void *stream);
int dllm_cluster_select(const float *C_now, const float *C_prev, const int32_t *assign, int kc, int32_t *idx,
                        int32_t *count, int B, int N, int D, int K, void *stream);

/* ---------------------------------------------------------------------------
 * Selection.  [SPA] "1. ...": the rows with the lowest proxy similarity (largest
 * drift) are recomputed, [SPA] "2. Adaptive budget allocation": at most k of them
 * per layer; [EC] step 3: the current masked tokens and the k most recently decoded
 * tokens are always recomputed (the forced set).
 *
 * For each sequence b:  F_b = entries of forced[b, 0..F) inside [0, N) (others are
 * padding; duplicates count once);  eligible = rows not in F_b with drift > min_drift
 * (NaN is never eligible);  the min(k, N - |F_b|) eligible rows with the largest
 * drift are taken, equal drifts by lower row index;  idx[b, 0..count[b]) receives
 * F_b union taken in ascending order and idx[b, count[b]..N) = -1.
 *   drift  [B, N] fp32;  forced [B, F] int32 or NULL (then F is ignored);
 *   idx    [B, N] int32 out;  count [B] int32 out.
 * Requirements: N <= 16384, 0 <= k.  No workspace.
 * ------------------------------------------------------------------------- */
int dllm_select_topk(const float *drift, const int32_t *forced, int F, int k, float min_drift,
                     int32_t *idx, int32_t *count, int B, int N, void *stream);

/* Per-layer update ratio, [SPA] "2. Adaptive budget allocation" (a piecewise Gaussian
 * over depth): rho(l) = base + (peak - base) exp(-(l - centre)^2 / (2 s^2)) with
 * s = sigma_left below the centre and sigma_right from it on.  Host function. */
double dllm_layer_rho(int l, double base, double peak, double centre, double sigma_left,
                      double sigma_right);

/* Drift budget of a layer: ceil(rho * N), at least 1 when rho > 0, at most N.  Host. */
int dllm_layer_budget(double rho, int N);

/* ---------------------------------------------------------------------------
 * Layer weights.  nn.Linear layout in ([out, in]) is repacked once per layer:
 *   w_qkv  [(n_q + 2 n_kv) hd, d]  rows Q | K | V; inside every head the rows are
 *          ordered 0, hd/2, 1, hd/2+1, ... so that the two halves of each rotary pair
 *          are neighbours (outputs are written back in the natural order);
 *   w_o    [d, n_q hd];   w_gu [2F, d] with row 2j = gate j, row 2j+1 = up j;
 *   w_down [d, F];        gamma1, gamma2 [d];  rope_inv_freq [hd/2] fp32.
 * ------------------------------------------------------------------------- */
typedef struct dllm_layer {
    const void *w_qkv;
    const void *w_o;
    const void *w_gu;
    const void *w_down;
    const void *gamma1;
    const void *gamma2;
    const float *rope_inv_freq; /* [hd/2] fp32: rope_theta^(-2i/hd), built in double */
    int d, n_q, n_kv, hd, F;
    float eps;        /* RMSNorm epsilon                                     */
    float rope_theta; /* rotary base                                          */
    int use_rope;     /* 1: rotate Q and K (rotate-half pairs) at their rows  */
    int dtype;        /* DLLM_BF16 or DLLM_F32                               */
} dllm_layer;

/* Bytes of packed weights for one layer (256-byte aligned sub-buffers). */
size_t dllm_packed_layer_bytes(int d, int n_q, int n_kv, int hd, int F, int dtype);

/* Repacks one layer's nn.Linear weights (device, dtype) into dst and fills *out with
 * pointers into dst.  Sources may be freed once the stream has run the copy.
 * Requirements: hd in {64, 128}; n_q % n_kv == 0; d, n_q hd, F multiples of 64 for
 * DLLM_BF16 (of 2 for DLLM_F32). */
int dllm_pack_layer(const void *w_q, const void *w_k, const void *w_v, const void *w_o,
                    const void *w_g, const void *w_u, const void *w_d, const void *gamma1,
                    const void *gamma2, int d, int n_q, int n_kv, int hd, int F, float eps,
                    float rope_theta, int use_rope, int dtype, void *dst, size_t dst_bytes,
                    dllm_layer *out, void *stream);

/* ---------------------------------------------------------------------------
 * [SPA] "3. Sparse execution": recompute only the selected rows.
 *
 * For every sequence b and selected row i = idx[b, s], s < min(count[b], k_max):
 *   xn = RMSNorm(H_in[b,i]) gamma1;  q, k, v = xn W_q^T, xn W_k^T, xn W_v^T;
 *   rotary embedding of q and k at position i (rotate-half, base rope_theta);
 *   K_cache[b,i] <- k, V_cache[b,i] <- v          (all selected rows first, so the
 *                                                   queries see the partially updated cache)
 *   a = softmax(q K_cache[b]^T / sqrt(hd)) V_cache[b] over all N rows (non-causal;
 *       query head h reads KV head h / (n_q / n_kv));
 *   h1 = H_in[b,i] + a W_o^T;  x2 = RMSNorm(h1) gamma2;
 *   H_out_cache[b,i] <- h1 + (SiLU(x2 W_g^T) * (x2 W_u^T)) W_down^T;
 *   proxy_cache[b,i] <- proxy_cur[b,i]              (when both pointers are non-NULL).
 * Rows that are not selected are not written.
 *   H_in        [B, N, d]        dtype
 *   idx, count  as written by dllm_select_topk ([B, N] and [B] int32)
 *   k_max       host upper bound on count[b]; larger counts are clamped and flagged
 *   K_cache, V_cache [B, N, n_kv, hd] dtype (in/out); H_out_cache [B, N, d] dtype (in/out)
 *   proxy_cache, proxy_cur [B, N, r] fp32 or NULL
 * Requirements: k_max <= N; H_out_cache must not alias H_in.
 * ------------------------------------------------------------------------- */
size_t dllm_refresh_workspace_bytes(const dllm_layer *W, int B, int N, int k_max);

int dllm_sparse_layer_refresh(const dllm_layer *W, const void *H_in, const int32_t *idx,
                              const int32_t *count, int k_max, void *K_cache, void *V_cache,
                              void *H_out_cache, float *proxy_cache, const float *proxy_cur, int r,
                              int B, int N, void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * One layer's sparse step in one call: [SPA] "1. Update identification via singular
 * proxy" (dllm_proxy_score on H_in), "2. Adaptive budget allocation" with [EC] "How
 * EntropyCache works" step 3 (dllm_select_topk with the forced rows and the budget k),
 * "3. Sparse execution" (dllm_sparse_layer_refresh of the selected rows with
 * k_max = min(N, k + F)).  The outputs are those of the three calls in sequence:
 *   proxy_cur, drift                       as dllm_proxy_score (proxy_cache is its cache)
 *   idx, count                             as dllm_select_topk
 *   K_cache, V_cache, H_out_cache, proxy_cache   as dllm_sparse_layer_refresh
 * The selection is fused with the gather of the selected rows for N <= 4096 (one kernel
 * fewer, no host round trip between the steps); longer sequences run the separate
 * kernels.  For bf16 with r <= 128 and a proxy projection that splits K, that kernel also
 * sums the projection's partials and computes the drift (no cosine kernel): its CTAs of a
 * sequence wait for one another at an arrival counter in the workspace (bounded: after
 * 1 s the wait gives up and raises DLLM_STATUS_TIMEOUT), which the launch takes only when
 * the whole grid fits the GPU at once, and otherwise keeps the cosine kernel.  Results
 * are the same either way.  Pt [r, d] in the layer's dtype; forced [B, F] int32 (-1
 * padded) or NULL.
 * Requirements: those of the three calls (r % 32 == 0; N <= 16384; H_out_cache not
 * aliasing H_in; 16-byte aligned arrays).  Workspace:
 * dllm_layer_step_workspace_bytes(W, B, N, r, F, k) bytes.
 * ------------------------------------------------------------------------- */
size_t dllm_layer_step_workspace_bytes(const dllm_layer *W, int B, int N, int r, int F, int k);

int dllm_layer_step(const dllm_layer *W, const void *Pt, const void *H_in, float *proxy_cache,
                    float *proxy_cur, float *drift, const int32_t *forced, int F, int k, float min_drift,
                    int32_t *idx, int32_t *count, void *K_cache, void *V_cache, void *H_out_cache,
                    int B, int N, int r, void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * Vocabulary step.  [TSPD] "Input features": top-1 confidence and predictive entropy
 * per token; [EC] step 2: the maximum entropy E of the tokens decoded at this step,
 * step 3: E > tau means a full forward at the next step; [POL] "1. Problem
 * definition" / [TSPD]: static confidence-threshold commit.
 *
 * For every row (b, m) with valid[b, m] != 0, p = softmax(logits[b, m]):
 *   conf = max p, entropy = -sum p ln p (nats), argmax = lowest id of the maximum.
 * Per sequence: commit every valid row with conf >= conf_thresh; if none qualifies,
 * commit the one valid row with the highest conf (lowest m on ties);
 *   token[b, m] = argmax of committed rows, -1 otherwise;
 *   max_entropy[b] = max entropy over committed rows (0 if none);
 *   full_next[b] = max_entropy[b] > tau.
 * conf and entropy of invalid rows are 0.
 *   logits [B, M, V] fp32;  valid [B, M] uint8;  token [B, M] int32 out;
 *   conf, entropy [B, M] fp32 out;  max_entropy [B] fp32 out;  full_next [B] int32 out.
 * Requirements: M <= 1024, V >= 1.
 * ------------------------------------------------------------------------- */
size_t dllm_commit_workspace_bytes(int B, int M, int V);

int dllm_commit_entropy(const float *logits, const uint8_t *valid, int B, int M, int V,
                        float conf_thresh, float tau, int32_t *token, float *conf,
                        float *entropy, float *max_entropy, int32_t *full_next, void *ws,
                        size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * LM head fused with the vocabulary step ([EC] step 2, [TSPD] "Input features"): the
 * same outputs as dllm_commit_entropy on logits = X W_lm^T, without materialising the
 * logits.  The product runs on the tensor cores and reduces each 128-row tile of the
 * vocabulary to one online-softmax state (max, argmax, sum of exponentials, their
 * weighted sum) per row, which the commit step merges in a fixed order.
 *   X [B*M, d] bf16 (the block rows after the final RMSNorm, as dllm_rows_rmsnorm
 *   writes them), W_lm [V, d] bf16, valid [B, M] uint8; outputs as dllm_commit_entropy.
 * Requirements: M <= 1024, d % 64 == 0, V % 32 == 0.  Workspace:
 * dllm_lmhead_workspace_bytes(B, M, V) bytes (16 bytes per row and vocabulary tile).
 * ------------------------------------------------------------------------- */
size_t dllm_lmhead_workspace_bytes(int B, int M, int V);

int dllm_lmhead_commit(const void *X, const void *W_lm, const uint8_t *valid, int B, int M, int V,
                       int d, float conf_thresh, float tau, int32_t *token, float *conf,
                       float *entropy, float *max_entropy, int32_t *full_next, void *ws,
                       size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * [SPA] "3. Sparse execution", the attention of the selected queries alone (the same
 * kernels dllm_sparse_layer_refresh runs after the K/V scatter):
 *   A[m, h] = softmax(Q[m, h] K_cache[b, :, g]^T / sqrt(hd)) V_cache[b, :, g]
 * over all N rows, non-causal, g = h / (n_q / n_kv), for every flattened row
 * m = b * k_max + s that is live (s < min(count[b], k_max) and idx[b, s] in [0, N));
 * other rows of A get zeros.  Q and A [B*k_max, n_q*hd]; K_cache, V_cache [B, N, n_kv, hd];
 * idx [B, N], count [B] int32 as written by dllm_select_topk; dtype as the caches.
 * Requirements: hd in {64, 128}; k_max <= N.
 * Workspace: dllm_attention_workspace_bytes() bytes (currently 0 for every shape: the
 * key-range split is merged on chip); ws may then be NULL.
 * ------------------------------------------------------------------------- */
size_t dllm_attention_workspace_bytes(int B, int N, int k_max, int n_q, int hd, int dtype);

int dllm_attention(const void *Q, const void *K_cache, const void *V_cache, void *A,
                   const int32_t *idx, const int32_t *count, int k_max, int B, int N, int n_q,
                   int n_kv, int hd, int dtype, void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * dllm_commit_entropy without a workspace.  (No counterpart on the pages: this is an
 * interface variant, not a step of the method.)
 *
 * For callers that cannot allocate device memory themselves -- for example code that
 * only receives device buffers from a host application and has no cudaMalloc or
 * caching allocator of its own -- this entry point keeps its scratch (one softmax
 * state per row slice) in a fixed device array inside the library instead of a
 * caller workspace, and allocates nothing: no cudaMalloc, no cudaFree, no allocating
 * library routine.  The array holds 16384 states (256 KB) and stays resident on every
 * GPU that loads the library until the process exits; shapes that need more (roughly
 * B*M rows x ceil(V/2048) slices, capped by the GPU size) are rejected with
 * DLLM_ERR_UNSUPPORTED and a message.  Outputs, arguments and results are those of
 * dllm_commit_entropy.
 * The first call on a device looks up the array's device address (once per device,
 * with that device current); make that first call before any stream capture.  All
 * calls share the one array and it keeps the previous call's contents (each call
 * writes every state it reads, so nothing needs clearing); calls whose kernels could
 * overlap on the GPU (different streams without ordering) race on it.
 * ------------------------------------------------------------------------- */
int dllm_commit_entropy_noalloc(const float *logits, const uint8_t *valid, int B, int M, int V,
                                float conf_thresh, float tau, int32_t *token, float *conf,
                                float *entropy, float *max_entropy, int32_t *full_next,
                                void *stream);

/* ---------------------------------------------------------------------------
 * Around the layers of a denoising step ([EC] step 1: the forward pass; step 2:
 * decode from the logits of the current block).
 *
 * dllm_embed: H[b, i] = E[tokens[b, i]] for every i (rows == NULL) or for the R
 *   positions rows[b, 0..R) (entries outside [0, N) skipped); token ids outside
 *   [0, V) give a zero row.  E [V, d], tokens [B, N] int32, H [B, N, d], dtype.
 * dllm_rows_rmsnorm: out[b*R + j] = RMSNorm(H[b, rows[b, j]]) * gamma (zeros for
 *   entries outside [0, N)): the final norm of the rows fed to the LM head.
 *   H [B, N, d], rows [B, R] int32, gamma [d], out [B*R, d], dtype.
 * ------------------------------------------------------------------------- */
int dllm_embed(const void *E, const int32_t *tokens, const int32_t *rows, int R, void *H, int B,
               int N, int d, int V, int dtype, void *stream);

int dllm_rows_rmsnorm(const void *H, const int32_t *rows, int R, const void *gamma, float eps,
                      void *out, int B, int N, int d, int dtype, void *stream);

/* ---------------------------------------------------------------------------
 * [SPA] "3. Sparse execution": the rows a refresh rewrote, packed for the caller (the
 * refreshed hidden states, keys or values that leave the device after a step):
 *   dst[b * k_max + s] = src[b, idx[b, s]]   for s < min(count[b], k_max) and
 *                                            idx[b, s] in [0, N);
 *   dst[b * k_max + s] = 0 bytes             for the other rows.
 * src [B, N, row_bytes] bytes (H_out_cache rows: row_bytes = d * element size; K/V cache
 * rows: n_kv * hd * element size), dst [B * k_max, row_bytes]; idx [B, N] and count [B]
 * int32 as written by dllm_select_topk.  Requirements: row_bytes % 16 == 0, src and dst
 * 16-byte aligned, 0 < k_max <= N.  No workspace.  Errors: INVALID_ARG (null pointer,
 * sizes, alignment), CUDA (launch).
 * ------------------------------------------------------------------------- */
int dllm_gather_rows(const void *src, const int32_t *idx, const int32_t *count, int k_max, void *dst,
                     int B, int N, int row_bytes, void *stream);

/* The same packing for n <= 4 caches that share one selection, in one launch (a step's
 * refreshed H_out, K and V rows): for t < n, dsts[t] [B * k_max, row_bytes[t]] receives the
 * rows of srcs[t] [B, N, row_bytes[t]] as dllm_gather_rows would.  srcs, dsts and
 * row_bytes are host arrays of n entries (read during the call); the pointers they hold
 * are device pointers.  Requirements and errors as dllm_gather_rows, per cache; n outside
 * [1, 4] is INVALID_ARG. */
int dllm_gather_rows_n(int n, const void *const *srcs, void *const *dsts, const int *row_bytes,
                       const int32_t *idx, const int32_t *count, int k_max, int B, int N, void *stream);

/* ---------------------------------------------------------------------------
 * Plain product on the tensor cores, the engine under every bf16 projection above
 * (and the LM head of the vocabulary step: logits = RMSNorm(h) W_lm^T):
 *   out[m, f] = sum_k X[m, k] W[f, k]          (fp32 accumulation and output)
 *   X [M, K] bf16, W [N_out, K] bf16 (nn.Linear layout), out [M, N_out] fp32.
 * splits: number of CTAs that share one output tile along K (a thread-block cluster
 * reducing through distributed shared memory); 0 = chosen from the shape, 1..8.
 * Requirements: K % 64 == 0, N_out % 32 == 0, 16-byte aligned rows.  No workspace.
 * ------------------------------------------------------------------------- */
int dllm_gemm_bf16(const void *X, const void *W, float *out, int M, int N_out, int K, int splits,
                   void *stream);

/* The launch plan dllm_gemm_bf16 (slices = 0), the proxy projection's independent K
 * slices (slices = 1) or the proxy projection with its drift in the epilogue (slices = 2,
 * N_out = r <= 128; dllm_proxy_score takes it when the slice plan has no K split) would
 * use for this shape on a device with `sms` SMs.  Host only:
 * no device is queried and nothing is launched, so it answers without a GPU (the
 * library's own launches pass the current device's SM count).  info [8] receives
 *   { token-tile width BN, K split, pipeline stages, token tiles, weight tiles of 128
 *     rows, token rows staged per K block, dynamic shared memory bytes, CTAs per SM }.
 * splits as for dllm_gemm_bf16 (0 = chosen from the shape).  Errors: INVALID_ARG for a
 * null info, sizes <= 0, sms outside [1, 1024], splits outside [0, 8], slices outside
 * [0, 2] or slices = 2 with N_out > 128; UNSUPPORTED when K % 64 or N_out % 32 is not 0. */
int dllm_gemm_plan(int M, int N_out, int K, int splits, int sms, int slices, int32_t *info);

/* ---------------------------------------------------------------------------
 * Measurement support.  While a timer is armed, every launch of the chosen kernel
 * (any stream) is bracketed by a pair of CUDA events, up to max_launches launches;
 * dllm_timer_stop() synchronises the device, returns the summed event time and the
 * number of timed launches, and disarms.  dllm_launch_count() is the number of
 * kernels this library has launched in the process so far.
 * ------------------------------------------------------------------------- */
#define DLLM_KERNEL_PROXY_GEMM 1
#define DLLM_KERNEL_COSINE 2
#define DLLM_KERNEL_SELECT 3
#define DLLM_KERNEL_GATHER 4
#define DLLM_KERNEL_QKV 5
#define DLLM_KERNEL_ATTENTION 6
#define DLLM_KERNEL_OPROJ 7
#define DLLM_KERNEL_RMSNORM2 8
#define DLLM_KERNEL_GATEUP 9
#define DLLM_KERNEL_DOWN 10
#define DLLM_KERNEL_VOCAB 11
#define DLLM_KERNEL_GEMM 12
#define DLLM_KERNEL_KL_DRIFT 13
#define DLLM_KERNEL_CE 14
#define DLLM_KERNEL_POLESTAR 15
#define DLLM_KERNEL_CLUSTER 16

/* Launch mode of the library's kernels: with enable != 0 (the default) consecutive
 * kernels on a stream use programmatic dependent launch (a kernel's prologue and its
 * weight loads overlap the previous kernel's tail; it reads produced data only after
 * that kernel has completed).  Returns the previous setting.  Host function. */
int dllm_set_pdl(int enable);

int dllm_timer_start(int kernel_id, int max_launches);
int dllm_timer_stop(double *total_ms, int *launches);
unsigned long long dllm_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* DLLM_H_ */
