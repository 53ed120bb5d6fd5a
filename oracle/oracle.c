/*
 * oracle.c -- plain, slow CPU reference of the sparse KV-cache refresh step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg may load this file's library.  It shares no code, header,
 * table or helper with the CUDA library and includes nothing from it.
 *
 * Storage is fp32; every dot product, sum, norm and softmax accumulates in
 * double.  Per-row intermediates are kept in double.  Loops follow the order
 * in which the pages state the method; nothing is blocked, fused or reordered
 * beyond an OpenMP split over independent rows.
 *
 * Sources (page title, section):
 *  [SPA]  "Singular proxies for adaptive caching in diffusion language models"
 *         (SPA-Cache): "1. Update identification via singular proxy",
 *         "2. Adaptive budget allocation", "3. Sparse execution".
 *  [EC]   "EntropyCache": "How EntropyCache works" steps 1-3.
 *  [TSPD] "Temporal-Spatial Parallel Decoding and Confidence Extrapolation":
 *         "Input features" (top-1 confidence, predictive entropy).
 *  [POL]  "Polestar: drift-aware cache correction and token commit for efficient
 *         diffusion LLM inference": "1. Problem definition" (static
 *         confidence-threshold commit).
 *
 * Readings where the pages are silent are listed next to each function.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define EXPORT __attribute__((visibility("default")))

/* One bidirectional pre-norm transformer layer, weights in nn.Linear layout
 * [out_features, in_features], fp32. */
typedef struct {
    const float *w_q;    /* [n_q*hd, d]  */
    const float *w_k;    /* [n_kv*hd, d] */
    const float *w_v;    /* [n_kv*hd, d] */
    const float *w_o;    /* [d, n_q*hd]  */
    const float *w_g;    /* [F, d] gate  */
    const float *w_u;    /* [F, d] up    */
    const float *w_d;    /* [d, F] down  */
    const float *gamma1; /* [d] pre-attention RMSNorm gain */
    const float *gamma2; /* [d] pre-FFN RMSNorm gain */
    int d, n_q, n_kv, hd, F;
    float eps, rope_theta;
    int use_rope;
} oracle_layer;

static int g_threads = 1;

EXPORT void oracle_set_threads(int n) { g_threads = n > 0 ? n : 1; }

EXPORT int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_num_procs();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------- */
/* small dense helpers (double accumulation)                                  */
/* ------------------------------------------------------------------------- */

/* y[j] = sum_k W[j,k] * x[k]   (W row-major [rows, cols], nn.Linear orientation) */
static void linear(const float *W, const double *x, int rows, int cols, double *y) {
    for (int j = 0; j < rows; ++j) {
        const float *w = W + (size_t)j * cols;
        double acc = 0.0;
        for (int k = 0; k < cols; ++k) acc += (double)w[k] * x[k];
        y[j] = acc;
    }
}

/* RMSNorm: x / sqrt(mean(x^2) + eps) * gamma */
static void rmsnorm(const double *x, const float *gamma, int d, float eps, double *out) {
    double ss = 0.0;
    for (int k = 0; k < d; ++k) ss += x[k] * x[k];
    double inv = 1.0 / sqrt(ss / d + (double)eps);
    for (int k = 0; k < d; ++k) out[k] = x[k] * inv * (double)gamma[k];
}

/* Rotary embedding, rotate-half convention: the pair (x[i], x[i+hd/2]) is
 * rotated by the angle pos * theta^(-2i/hd). */
static void rope(double *x, int hd, int pos, double theta) {
    int half = hd / 2;
    for (int i = 0; i < half; ++i) {
        double freq = pow(theta, -2.0 * i / hd);
        double ang = pos * freq;
        double c = cos(ang), s = sin(ang);
        double x1 = x[i], x2 = x[i + half];
        x[i] = x1 * c - x2 * s;
        x[i + half] = x2 * c + x1 * s;
    }
}

/* One head vector rotated in place at position pos (exported for the pins). */
EXPORT void oracle_rope_row(float *x, int hd, int pos, float theta) {
    double *t = (double *)malloc(sizeof(double) * hd);
    for (int e = 0; e < hd; ++e) t[e] = x[e];
    rope(t, hd, pos, theta);
    for (int e = 0; e < hd; ++e) x[e] = (float)t[e];
    free(t);
}

static double silu(double x) { return x / (1.0 + exp(-x)); }

/* ------------------------------------------------------------------------- */
/* [SPA] "1. Update identification via singular proxy"                        */
/* ------------------------------------------------------------------------- */

/* Cosine drift between a current and a cached proxy vector:
 * drift = 1 - <s, c> / sqrt(<s,s> <c,c>), clamped to [0, 2].
 * Readings: both norms zero -> 0 (nothing changed); one norm zero -> 1. */
static double cosine_drift(const float *s, const float *c, int r) {
    double dot = 0.0, ns = 0.0, nc = 0.0;
    for (int j = 0; j < r; ++j) {
        dot += (double)s[j] * c[j];
        ns += (double)s[j] * s[j];
        nc += (double)c[j] * c[j];
    }
    if (ns == 0.0 && nc == 0.0) return 0.0;
    if (ns == 0.0 || nc == 0.0) return 1.0;
    double dr = 1.0 - dot / sqrt(ns * nc);
    if (dr < 0.0) dr = 0.0;
    if (dr > 2.0) dr = 2.0;
    return dr;
}

/* Singular proxy and drift score for every token.
 *   H [B, N, d] layer input, P [d, r] proxy matrix (top-r left singular vectors
 *   scaled by their singular values, built once per layer),
 *   proxy_cache [B, N, r] proxies stored when each row was last refreshed.
 * Outputs proxy_cur [B, N, r] = H P and drift [B, N]. */
EXPORT void oracle_proxy_score(const float *H, const float *P, const float *proxy_cache,
                               float *proxy_cur, float *drift, int B, int N, int d, int r) {
    long rows = (long)B * N;
#pragma omp parallel for schedule(static) num_threads(g_threads)
    for (long t = 0; t < rows; ++t) {
        const float *h = H + t * d;
        float *s = proxy_cur + t * r;
        for (int j = 0; j < r; ++j) {
            double acc = 0.0;
            for (int k = 0; k < d; ++k) acc += (double)h[k] * P[(size_t)k * r + j];
            s[j] = (float)acc;
        }
        drift[t] = (float)cosine_drift(s, proxy_cache + t * r, r);
    }
}

/* Drift score alone, from given current and cached proxies (fp32 inputs). */
EXPORT void oracle_cosine_drift(const float *cur, const float *cached, float *drift, long rows, int r) {
    for (long t = 0; t < rows; ++t) drift[t] = (float)cosine_drift(cur + t * r, cached + t * r, r);
}

/* ------------------------------------------------------------------------- */
/* Selection: [SPA] lowest similarity first under the layer budget;           */
/* [EC] step 3: current masked tokens and the k most recent decoded tokens    */
/* are always recomputed.                                                     */
/* ------------------------------------------------------------------------- */

/* For each sequence b:
 *   forced set F_b = valid entries of forced[b, 0..F) (entries < 0 or >= N are padding);
 *   eligible rows = not in F_b and drift > min_drift;
 *   take up to min(k, N - |F_b|) eligible rows by repeatedly picking the one with
 *   the largest drift (lower row index on equal drift);
 *   I_b = F_b union picked, written ascending to idx[b, 0..count[b]).
 * idx has row stride N.  NaN drift is never eligible. */
EXPORT void oracle_select_topk(const float *drift, const int32_t *forced, int F, int k,
                               float min_drift, int32_t *idx, int32_t *count, int B, int N) {
    unsigned char *in = (unsigned char *)malloc((size_t)N);
    for (int b = 0; b < B; ++b) {
        const float *dr = drift + (size_t)b * N;
        memset(in, 0, (size_t)N);
        int nforced = 0;
        for (int f = 0; f < F && forced; ++f) {
            int p = forced[(size_t)b * F + f];
            if (p >= 0 && p < N && !in[p]) { in[p] = 1; ++nforced; }
        }
        int budget = k < N - nforced ? k : N - nforced;
        if (budget < 0) budget = 0;
        for (int pick = 0; pick < budget; ++pick) {
            int best = -1;
            for (int i = 0; i < N; ++i) {
                if (in[i] || !(dr[i] > min_drift)) continue;
                if (best < 0 || dr[i] > dr[best]) best = i;   /* strict: lower index wins ties */
            }
            if (best < 0) break;
            in[best] = 2;
        }
        int c = 0;
        for (int i = 0; i < N; ++i)
            if (in[i]) idx[(size_t)b * N + c++] = i;
        for (int i = c; i < N; ++i) idx[(size_t)b * N + i] = -1;
        count[b] = c;
    }
    free(in);
}

/* [SPA] "2. Adaptive budget allocation": per-layer update ratio as a piecewise
 * Gaussian over depth (low early, peak in the middle, low late).
 * Reading: rho(l) = base + (peak - base) * exp(-(l - centre)^2 / (2 sigma^2)),
 * sigma = sigma_left for l < centre, sigma_right otherwise. */
EXPORT double oracle_rho(int l, double base, double peak, double centre, double sigma_left,
                         double sigma_right) {
    double s = (l < centre) ? sigma_left : sigma_right;
    double z = (l - centre) / s;
    return base + (peak - base) * exp(-0.5 * z * z);
}

/* Drift budget of a layer: ceil(rho * N) rows, at least 1 when rho > 0, at most N. */
EXPORT int oracle_budget(double rho, int N) {
    if (!(rho > 0.0)) return 0;
    double kk = ceil(rho * N);
    int k = (int)kk;
    if (k < 1) k = 1;
    if (k > N) k = N;
    return k;
}

/* ------------------------------------------------------------------------- */
/* [SPA] "3. Sparse execution"                                                */
/* ------------------------------------------------------------------------- */

/* Attention output of one query row q (already rotated) against all N rows of
 * one sequence's cache, for every head; softmax scale 1/sqrt(hd); non-causal.
 * Query head h reads key/value head h / (n_q / n_kv). */
static void attend_row(const oracle_layer *W, const double *q, const float *Kc, const float *Vc,
                       int N, double *a /* [n_q*hd] */, double *p /* [N] scratch */) {
    int hd = W->hd, group = W->n_q / W->n_kv, dkv = W->n_kv * hd;
    double scale = 1.0 / sqrt((double)hd);
    for (int h = 0; h < W->n_q; ++h) {
        int g = h / group;
        const double *qh = q + (size_t)h * hd;
        double mx = -INFINITY;
        for (int j = 0; j < N; ++j) {
            const float *kj = Kc + (size_t)j * dkv + (size_t)g * hd;
            double sc = 0.0;
            for (int e = 0; e < hd; ++e) sc += qh[e] * kj[e];
            p[j] = sc * scale;
            if (p[j] > mx) mx = p[j];
        }
        double z = 0.0;
        for (int j = 0; j < N; ++j) { p[j] = exp(p[j] - mx); z += p[j]; }
        double *ah = a + (size_t)h * hd;
        for (int e = 0; e < hd; ++e) ah[e] = 0.0;
        for (int j = 0; j < N; ++j) {
            const float *vj = Vc + (size_t)j * dkv + (size_t)g * hd;
            double w = p[j] / z;
            for (int e = 0; e < hd; ++e) ah[e] += w * vj[e];
        }
    }
}

/* Everything after attention for one row: O projection + residual, pre-FFN
 * RMSNorm, SwiGLU FFN + residual.  h_in is the layer input row. */
static void post_attention(const oracle_layer *W, const float *h_in, const double *a, float *out) {
    int d = W->d, dq = W->n_q * W->hd, F = W->F;
    double *o = (double *)malloc(sizeof(double) * d);
    double *h1 = (double *)malloc(sizeof(double) * d);
    double *xn2 = (double *)malloc(sizeof(double) * d);
    double *g = (double *)malloc(sizeof(double) * F);
    double *u = (double *)malloc(sizeof(double) * F);
    double *f = (double *)malloc(sizeof(double) * d);
    linear(W->w_o, a, d, dq, o);
    for (int k = 0; k < d; ++k) h1[k] = (double)h_in[k] + o[k];
    rmsnorm(h1, W->gamma2, d, W->eps, xn2);
    linear(W->w_g, xn2, F, d, g);
    linear(W->w_u, xn2, F, d, u);
    for (int j = 0; j < F; ++j) g[j] = silu(g[j]) * u[j];
    linear(W->w_d, g, d, F, f);
    for (int k = 0; k < d; ++k) out[k] = (float)(h1[k] + f[k]);
    free(o); free(h1); free(xn2); free(g); free(u); free(f);
}

/* Query/key/value of one row at position pos; keys and queries rotated. */
static void qkv_row(const oracle_layer *W, const float *h_in, int pos, double *q, double *kk, double *v) {
    int d = W->d, dq = W->n_q * W->hd, dkv = W->n_kv * W->hd;
    double *x = (double *)malloc(sizeof(double) * d);
    double *xn = (double *)malloc(sizeof(double) * d);
    for (int e = 0; e < d; ++e) x[e] = h_in[e];
    rmsnorm(x, W->gamma1, d, W->eps, xn);
    linear(W->w_q, xn, dq, d, q);
    linear(W->w_k, xn, dkv, d, kk);
    linear(W->w_v, xn, dkv, d, v);
    if (W->use_rope) {
        for (int h = 0; h < W->n_q; ++h) rope(q + (size_t)h * W->hd, W->hd, pos, W->rope_theta);
        for (int h = 0; h < W->n_kv; ++h) rope(kk + (size_t)h * W->hd, W->hd, pos, W->rope_theta);
    }
    free(x); free(xn);
}

/* Sparse refresh of one layer at the selected rows I_b = idx[b, 0..count[b]).
 *   1. for every i in I_b: q, k, v from RMSNorm(H_in[b,i]); k and v are written
 *      into K_cache[b,i], V_cache[b,i] (all of I_b before any attention, so the
 *      selected queries see the partially updated cache);
 *   2. for every i in I_b: attention of q_i over all N cache rows, O projection,
 *      residual, SwiGLU FFN, residual -> H_out_cache[b,i];
 *      proxy_cache[b,i] <- proxy_cur[b,i] (when both are given, r > 0).
 * Rows outside I_b are not touched.  idx has row stride idx_stride.
 * out_mask (optional, [B, N]): step 2 runs only for rows whose mask is non-zero
 * (sampled outputs for large shapes; step 1 always covers all of I_b). */
EXPORT void oracle_layer_refresh(const oracle_layer *W, const float *H_in, const int32_t *idx,
                                 const int32_t *count, int idx_stride, float *K_cache,
                                 float *V_cache, float *H_out_cache, float *proxy_cache,
                                 const float *proxy_cur, int r, int B, int N,
                                 const unsigned char *out_mask) {
    int d = W->d, dq = W->n_q * W->hd, dkv = W->n_kv * W->hd;
    for (int b = 0; b < B; ++b) {
        const int32_t *I = idx + (size_t)b * idx_stride;
        int c = count[b];
        const float *Hb = H_in + (size_t)b * N * d;
        float *Kb = K_cache + (size_t)b * N * dkv;
        float *Vb = V_cache + (size_t)b * N * dkv;
        double *Q = (double *)malloc(sizeof(double) * (size_t)(c > 0 ? c : 1) * dq);
#pragma omp parallel for schedule(dynamic) num_threads(g_threads)
        for (int s = 0; s < c; ++s) {
            int i = I[s];
            double *kk = (double *)malloc(sizeof(double) * dkv);
            double *v = (double *)malloc(sizeof(double) * dkv);
            qkv_row(W, Hb + (size_t)i * d, i, Q + (size_t)s * dq, kk, v);
            for (int e = 0; e < dkv; ++e) {
                Kb[(size_t)i * dkv + e] = (float)kk[e];
                Vb[(size_t)i * dkv + e] = (float)v[e];
            }
            free(kk); free(v);
        }
#pragma omp parallel for schedule(dynamic) num_threads(g_threads)
        for (int s = 0; s < c; ++s) {
            int i = I[s];
            if (out_mask && !out_mask[(size_t)b * N + i]) continue;
            double *a = (double *)malloc(sizeof(double) * dq);
            double *p = (double *)malloc(sizeof(double) * N);
            attend_row(W, Q + (size_t)s * dq, Kb, Vb, N, a, p);
            post_attention(W, Hb + (size_t)i * d, a, H_out_cache + ((size_t)b * N + i) * d);
            free(a); free(p);
        }
        if (proxy_cache && proxy_cur && r > 0)
            for (int s = 0; s < c; ++s) {
                size_t o = ((size_t)b * N + I[s]) * r;
                memcpy(proxy_cache + o, proxy_cur + o, sizeof(float) * r);
            }
        free(Q);
    }
}

/* Full (dense) forward of the layer over every row, written as its own loop:
 * the reference that a refresh of all rows must reproduce. */
EXPORT void oracle_layer_full(const oracle_layer *W, const float *H_in, float *K_cache,
                              float *V_cache, float *H_out, int B, int N) {
    int d = W->d, dq = W->n_q * W->hd, dkv = W->n_kv * W->hd;
    double *Q = (double *)malloc(sizeof(double) * (size_t)N * dq);
    for (int b = 0; b < B; ++b) {
        const float *Hb = H_in + (size_t)b * N * d;
        float *Kb = K_cache + (size_t)b * N * dkv;
        float *Vb = V_cache + (size_t)b * N * dkv;
#pragma omp parallel for schedule(static) num_threads(g_threads)
        for (int i = 0; i < N; ++i) {
            double *kk = (double *)malloc(sizeof(double) * dkv);
            double *v = (double *)malloc(sizeof(double) * dkv);
            qkv_row(W, Hb + (size_t)i * d, i, Q + (size_t)i * dq, kk, v);
            for (int e = 0; e < dkv; ++e) {
                Kb[(size_t)i * dkv + e] = (float)kk[e];
                Vb[(size_t)i * dkv + e] = (float)v[e];
            }
            free(kk); free(v);
        }
#pragma omp parallel for schedule(static) num_threads(g_threads)
        for (int i = 0; i < N; ++i) {
            double *a = (double *)malloc(sizeof(double) * dq);
            double *p = (double *)malloc(sizeof(double) * N);
            attend_row(W, Q + (size_t)i * dq, Kb, Vb, N, a, p);
            post_attention(W, Hb + (size_t)i * d, a, H_out + ((size_t)b * N + i) * d);
            free(a); free(p);
        }
    }
    free(Q);
}

/* Attention output rows alone (before the O projection), for pins on the
 * softmax: a[s, :] for query rows idx[0..c) of sequence 0 against its cache. */
EXPORT void oracle_attention_rows(const oracle_layer *W, const float *Q /* [c, n_q*hd] */,
                                  const float *K_cache, const float *V_cache, int N, int c,
                                  float *A /* [c, n_q*hd] */) {
    int dq = W->n_q * W->hd;
    double *q = (double *)malloc(sizeof(double) * dq);
    double *a = (double *)malloc(sizeof(double) * dq);
    double *p = (double *)malloc(sizeof(double) * N);
    for (int s = 0; s < c; ++s) {
        for (int e = 0; e < dq; ++e) q[e] = Q[(size_t)s * dq + e];
        attend_row(W, q, K_cache, V_cache, N, a, p);
        for (int e = 0; e < dq; ++e) A[(size_t)s * dq + e] = (float)a[e];
    }
    free(q); free(a); free(p);
}

/* ------------------------------------------------------------------------- */
/* Vocabulary side: [EC] step 2 (decode and maximum entropy), [TSPD] top-1    */
/* confidence and predictive entropy, [POL]/[TSPD] static threshold commit.   */
/* ------------------------------------------------------------------------- */

/* Final RMSNorm and LM head for M rows: logits[m, v] = <RMSNorm(h[m]) * gamma_f, W_lm[v]>. */
EXPORT void oracle_lmhead(const float *h, const float *gamma_f, const float *W_lm, int M, int d,
                          int V, float eps, float *logits) {
    for (int m = 0; m < M; ++m) {
        double *x = (double *)malloc(sizeof(double) * d);
        double *xn = (double *)malloc(sizeof(double) * d);
        for (int e = 0; e < d; ++e) x[e] = h[(size_t)m * d + e];
        rmsnorm(x, gamma_f, d, eps, xn);
#pragma omp parallel for schedule(static) num_threads(g_threads)
        for (int v = 0; v < V; ++v) {
            const float *w = W_lm + (size_t)v * d;
            double acc = 0.0;
            for (int e = 0; e < d; ++e) acc += (double)w[e] * xn[e];
            logits[(size_t)m * V + v] = (float)acc;
        }
        free(x); free(xn);
    }
}

/* Per-row distribution statistics of p = softmax(l):
 * argmax (lowest token id among equal maxima), p_max, entropy -sum p ln p (nats). */
EXPORT void oracle_vocab_stats(const float *logits, long rows, int V, int32_t *argmax,
                               float *pmax, float *entropy) {
#pragma omp parallel for schedule(static) num_threads(g_threads)
    for (long m = 0; m < rows; ++m) {
        const float *l = logits + (size_t)m * V;
        int am = 0;
        for (int v = 1; v < V; ++v)
            if (l[v] > l[am]) am = v;
        double mx = l[am];
        double z = 0.0;
        for (int v = 0; v < V; ++v) z += exp((double)l[v] - mx);
        double H = 0.0;
        for (int v = 0; v < V; ++v) {
            double p = exp((double)l[v] - mx) / z;
            if (p > 0.0) H -= p * log(p);
        }
        argmax[m] = am;
        pmax[m] = (float)(1.0 / z);   /* the maximum has exp(0) = 1 */
        entropy[m] = (float)H;
    }
}

/* Commit rule and full-refresh decision for each sequence b (rows m < M with valid[b,m]):
 *   commit every row with p_max >= conf_thresh; if none qualifies, commit the one row
 *   with the highest p_max (lowest row index on ties)  -- static threshold commit;
 *   E_b = maximum entropy over the rows committed at this step  -- [EC] step 2;
 *   full_next_b = (E_b > tau)  -- [EC] step 3 (E <= tau keeps the partial refresh).
 * token[b,m] = argmax for committed rows, -1 otherwise.  With no valid row, nothing
 * is committed, E_b = 0 and full_next_b = 0. */
EXPORT void oracle_commit_rule(const int32_t *argmax, const float *pmax, const float *entropy,
                               const unsigned char *valid, int B, int M, float conf_thresh,
                               float tau, int32_t *token, float *max_entropy, int32_t *full_next) {
    for (int b = 0; b < B; ++b) {
        int any = 0, best = -1;
        for (int m = 0; m < M; ++m) {
            size_t o = (size_t)b * M + m;
            token[o] = -1;
            if (!valid[o]) continue;
            if (pmax[o] >= conf_thresh) { token[o] = argmax[o]; any = 1; }
            if (best < 0 || pmax[o] > pmax[(size_t)b * M + best]) best = m;
        }
        if (!any && best >= 0) token[(size_t)b * M + best] = argmax[(size_t)b * M + best];
        double E = 0.0;
        int first = 1;
        for (int m = 0; m < M; ++m) {
            size_t o = (size_t)b * M + m;
            if (token[o] < 0) continue;
            if (first || entropy[o] > E) E = entropy[o];
            first = 0;
        }
        max_entropy[b] = (float)E;
        full_next[b] = (E > tau) ? 1 : 0;
    }
}

/* Whole vocabulary step on logits [B, M, V]: statistics of every valid row, then the
 * commit rule.  conf/entropy of invalid rows are 0. */
EXPORT void oracle_commit_entropy(const float *logits, const unsigned char *valid, int B, int M,
                                  int V, float conf_thresh, float tau, int32_t *token, float *conf,
                                  float *entropy, float *max_entropy, int32_t *full_next) {
    long rows = (long)B * M;
    int32_t *am = (int32_t *)malloc(sizeof(int32_t) * (rows > 0 ? rows : 1));
    oracle_vocab_stats(logits, rows, V, am, conf, entropy);
    for (long m = 0; m < rows; ++m)
        if (!valid[m]) { conf[m] = 0.0f; entropy[m] = 0.0f; }
    oracle_commit_rule(am, conf, entropy, valid, B, M, conf_thresh, tau, token, max_entropy,
                       full_next);
    free(am);
}
