/*
 * uno_oracle.c -- plain fp64 CPU oracle for the Uno draft+verify hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no source, header, table or helper with
 * the CUDA path.  It is deliberately slow and obvious: fp64 throughout, plain
 * loops, no blocking, no fusion, glibc exp/log, built without fast-math and
 * without FP contraction.  OpenMP only spreads independent rows/sequences
 * over host threads; it does not change any arithmetic.
 *
 * Pages cited (by title):
 *   [Explainer] "Unlocking Lossless Speedups in LLMs via Discrete Diffusion"
 *               (aifromscratch.in explainer)
 *   [Article]   "Uno Uses Discrete Diffusion to Accelerate LLMs Without Loss"
 *               (cctest.ai)
 *   [Summary]   "Unlocking Lossless Speedups in LLMs via Discrete Diffusion"
 *               (aiany.app summary)
 *
 * Functions and what pins them (the pins live in tests/, marked "not gpu"):
 *   oracle_gated_lora_linear_f64 -- [Explainer] "Two Decoupled Weight Sets":
 *       draft rows use theta_AR + theta_Delta (rank-128, alpha=256 LoRA),
 *       verification rows use theta_AR only.  Pinned by a hand-worked golden
 *       example, by numpy matmul for gate-0 rows, by the merged-weight form
 *       x.(W + (alpha/r) B A)^T for gate-1 rows, and by alpha=0 / B=0.
 *   oracle_verify_block_f64 -- [Explainer] "The Psi-Spec Sampler" (the drafts
 *       are rejection-sampled against the AR model; the accepted run ends at
 *       the first rejection; emitted tokens follow the AR model's
 *       distribution); [Article] "What 'lossless' means here".  Pinned by
 *       q==p => all accepted, disjoint supports => none accepted, the closed
 *       form E[n] = sum_k prod_{i<k} alpha_i, the acceptance threshold placed
 *       at min(1, p/q), and chi-square tests of the emitted tokens against p.
 *   oracle_draft_sample_f64 -- [Explainer] "The Psi-Spec Sampler" (the linear
 *       sampler draws a single token at each position).  Pinned by chi-square
 *       against softmax(logits).
 *
 * Readings where the pages are silent (the plainest reading in each case):
 *   - LoRA scale alpha/rank; layouts W[d_out,d_in], A[rank,d_in], B[d_out,rank].
 *   - Temperature 1 on the raw logits.
 *   - Accept draft i iff u_i < min(1, p_i(x_i)/q_i(x_i)), u_i in [0,1).
 *   - The residual max(0, p-q) (or p at a bonus position) is sampled by the
 *     exponential race: token = argmax_v r(v) / (-ln u_v), lowest v on a tie.
 *     With -ln u_v i.i.d. Exp(1) this picks v with probability r(v)/sum(r).
 *   - A sequence with a draft id outside [0,V) or a NaN/+inf logit (or a row
 *     that is -inf everywhere) gets a nonzero status, n=0 and no tokens.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_OK 0
#define OR_ERR_ARG (-1)
#define OR_ERR_NOMEM (-6)

/* per-sequence status codes (same meaning as the product library's) */
#define OR_SEQ_OK 0
#define OR_SEQ_BAD_DRAFT 1
#define OR_SEQ_NONFINITE 2

/* ------------------------------------------------------------------------ */
/* Gated-LoRA linear projection.                                            */
/*   y[m,n] = sum_k x[m,k] W[n,k]                                           */
/*          + g[m] * (alpha/rank) * sum_j (sum_k x[m,k] A[j,k]) B[n,j]       */
/* [Explainer] "Two Decoupled Weight Sets": rows of the draft pathway get   */
/* theta_AR plus the adapter (gate 1); verification rows get theta_AR alone  */
/* (gate 0).                                                                 */
/* All inputs are already fp64 (bf16/fp32 values widen exactly).            */
/* ------------------------------------------------------------------------ */
int oracle_gated_lora_linear_f64(const double *x, const double *W,
                                 const double *A, const double *B,
                                 const uint8_t *gate, int64_t M, int64_t d_in,
                                 int64_t d_out, int64_t rank, double alpha,
                                 double *y)
{
    if (M < 0 || d_in < 0 || d_out < 0 || rank < 0) return OR_ERR_ARG;
    if (M == 0 || d_out == 0) return OR_OK;
    if (!x || !W || !gate || !y) return OR_ERR_ARG;
    if (rank > 0 && (!A || !B)) return OR_ERR_ARG;
    const double scale = rank > 0 ? alpha / (double)rank : 0.0;
    int err = OR_OK;

#pragma omp parallel
    {
        double *t = (double *)malloc(sizeof(double) * (size_t)(rank > 0 ? rank : 1));
        if (!t) {
#pragma omp atomic write
            err = OR_ERR_NOMEM;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t m = 0; m < M; ++m) {
            if (!t) continue;
            const double *xm = x + m * d_in;
            /* LoRA down-projection of this row: t = x_m . A^T */
            for (int64_t j = 0; j < rank; ++j) {
                double s = 0.0;
                for (int64_t k = 0; k < d_in; ++k) s += xm[k] * A[j * d_in + k];
                t[j] = s;
            }
            const double g = (double)gate[m];
            for (int64_t n = 0; n < d_out; ++n) {
                double base = 0.0;
                for (int64_t k = 0; k < d_in; ++k) base += xm[k] * W[n * d_in + k];
                double lora = 0.0;
                for (int64_t j = 0; j < rank; ++j) lora += t[j] * B[n * rank + j];
                y[m * d_out + n] = base + g * scale * lora;
            }
        }
        free(t);
    }
    return err;
}

/* ------------------------------------------------------------------------ */
/* Softmax at temperature 1, fp64, max-subtracted, two passes.              */
/* Returns 0 on success, 1 if the row holds NaN or +inf or is all -inf.     */
/* ------------------------------------------------------------------------ */
static int softmax_row_f64(const float *logits, int64_t V, double *prob)
{
    double m = -INFINITY;
    for (int64_t v = 0; v < V; ++v) {
        const double l = (double)logits[v];
        if (isnan(l) || (isinf(l) && l > 0)) return 1;
        if (l > m) m = l;
    }
    if (isinf(m)) return 1; /* every entry is -inf: no distribution */
    double z = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        prob[v] = exp((double)logits[v] - m);
        z += prob[v];
    }
    for (int64_t v = 0; v < V; ++v) prob[v] /= z;
    return 0;
}

/* Exponential race: argmax_v w[v] / (-ln u[v]), lowest v on an exact tie.
 * With E_v = -ln u_v i.i.d. Exp(1), P(v wins) = w[v] / sum(w).
 * *margin receives (s1 - s2) / s1 for the two largest scores (+inf if only
 * one candidate has positive weight). */
static int32_t race_f64(const double *w, const float *u, int64_t V, double *margin)
{
    int32_t best = -1;
    double s1 = -1.0, s2 = -1.0;
    for (int64_t v = 0; v < V; ++v) {
        const double e = -log((double)u[v]);
        const double s = w[v] / e;
        if (s > s1) {
            s2 = s1;
            s1 = s;
            best = (int32_t)v;
        } else if (s > s2) {
            s2 = s;
        }
    }
    if (margin) *margin = (s2 > 0.0 && s1 > 0.0) ? (s1 - s2) / s1 : INFINITY;
    return best;
}

/* ------------------------------------------------------------------------ */
/* Block verifier (Psi-Spec linear sampler, verification half).             */
/* [Explainer] "The Psi-Spec Sampler": a block drafted in parallel is       */
/* checked against the AR model by rejection sampling (as in speculative    */
/* decoding); drafts are kept up to the first rejection and the emitted     */
/* tokens follow the AR model's distribution.  [Article] "What 'lossless'   */
/* means here": the AR model has the final say over every draft.            */
/*                                                                          */
/* p_logits [Bn,Kp,V] (AR, Kp = K or K+1), q_logits [Bn,K,V] (draft),       */
/* draft [Bn,K], u_acc [Bn,K] in [0,1), u_res [Bn,V] in (0,1).              */
/* Outputs n_accepted [Bn], out_tokens [Bn,K+1] (-1 padded), n_emitted [Bn],*/
/* status [Bn].  Optional: accept_margin [Bn,K] = |min(1,rho_i) - u_i| for  */
/* every evaluated position (+inf elsewhere), race_margin [Bn] (+inf when   */
/* no race ran).                                                            */
/* ------------------------------------------------------------------------ */
int oracle_verify_block_f64(const float *p_logits, const float *q_logits,
                            const int32_t *draft, const float *u_acc,
                            const float *u_res, int64_t Bn, int64_t K,
                            int64_t Kp, int64_t V, int32_t *n_accepted,
                            int32_t *out_tokens, int32_t *n_emitted,
                            int32_t *status, double *accept_margin,
                            double *race_margin)
{
    if (Bn < 0 || K < 0 || V <= 0 || (Kp != K && Kp != K + 1)) return OR_ERR_ARG;
    if (Bn == 0) return OR_OK;
    if (!p_logits || (K > 0 && (!q_logits || !draft || !u_acc)) || !u_res ||
        !n_accepted || !out_tokens || !n_emitted || !status)
        return OR_ERR_ARG;
    int err = OR_OK;

#pragma omp parallel
    {
        double *P = (double *)malloc(sizeof(double) * (size_t)(Kp > 0 ? Kp : 1) * (size_t)V);
        double *Q = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1) * (size_t)V);
        double *r = (double *)malloc(sizeof(double) * (size_t)V);
        if (!P || !Q || !r) {
#pragma omp atomic write
            err = OR_ERR_NOMEM;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t b = 0; b < Bn; ++b) {
            if (!P || !Q || !r) continue;
            int32_t *out = out_tokens + b * (K + 1);
            for (int64_t i = 0; i <= K; ++i) out[i] = -1;
            if (accept_margin)
                for (int64_t i = 0; i < K; ++i) accept_margin[b * K + i] = INFINITY;
            if (race_margin) race_margin[b] = INFINITY;
            n_accepted[b] = 0;
            n_emitted[b] = 0;
            status[b] = OR_SEQ_OK;

            /* Step 0: argument checks that belong to the sequence. */
            for (int64_t i = 0; i < K; ++i) {
                const int32_t x = draft[b * K + i];
                if (x < 0 || x >= V) status[b] = OR_SEQ_BAD_DRAFT;
            }
            /* Step 1: softmax of every AR row and every draft row. */
            int bad = 0;
            for (int64_t i = 0; i < Kp; ++i)
                bad |= softmax_row_f64(p_logits + (b * Kp + i) * V, V, P + i * V);
            for (int64_t i = 0; i < K; ++i)
                bad |= softmax_row_f64(q_logits + (b * K + i) * V, V, Q + i * V);
            if (bad && status[b] == OR_SEQ_OK) status[b] = OR_SEQ_NONFINITE;
            if (status[b] != OR_SEQ_OK) continue;

            /* Step 2: accept x_i iff u_i < min(1, p_i(x_i)/q_i(x_i)); stop at
             * the first rejection. */
            int64_t n = 0;
            for (int64_t i = 0; i < K; ++i) {
                const int32_t x = draft[b * K + i];
                const double pi = P[i * V + x];
                const double qi = Q[i * V + x];
                const double rho = qi > 0.0 ? pi / qi : INFINITY;
                const double thr = rho < 1.0 ? rho : 1.0;
                const double u = (double)u_acc[b * K + i];
                if (accept_margin) accept_margin[b * K + i] = fabs(thr - u);
                if (u < thr) {
                    out[i] = x;
                    ++n;
                } else {
                    break;
                }
            }
            n_accepted[b] = (int32_t)n;
            n_emitted[b] = (int32_t)n;

            /* Step 3: at the first rejection, sample from the normalised
             * residual max(0, p_n - q_n); if every draft was accepted and an
             * extra AR row exists, sample the bonus token from p_K. */
            const float *ub = u_res + b * V;
            double *rm = race_margin ? race_margin + b : NULL;
            if (n < K) {
                double S = 0.0;
                for (int64_t v = 0; v < V; ++v) {
                    const double d = P[n * V + v] - Q[n * V + v];
                    r[v] = d > 0.0 ? d : 0.0;
                    S += r[v];
                }
                if (S == 0.0) /* p_n == q_n: cannot happen after a rejection */
                    for (int64_t v = 0; v < V; ++v) r[v] = P[n * V + v];
                out[n] = race_f64(r, ub, V, rm);
                n_emitted[b] = (int32_t)(n + 1);
            } else if (Kp == K + 1) {
                out[K] = race_f64(P + K * V, ub, V, rm);
                n_emitted[b] = (int32_t)(K + 1);
            }
        }
        free(P);
        free(Q);
        free(r);
    }
    return err;
}

/* ------------------------------------------------------------------------ */
/* Sampling variants of the verifier: temperature and a single-uniform      */
/* inverse-CDF resample.  [Explainer] "The Psi-Spec Sampler": the           */
/* acceptance rule of speculative decoding, with every distribution taken   */
/* at sampling temperature T (p = softmax(l_p / T), q = softmax(l_q / T);   */
/* the drafts are assumed drawn from q at the same T).                      */
/* ------------------------------------------------------------------------ */
static int softmax_row_temp_f64(const float *logits, int64_t V, double T, double *prob)
{
    double m = -INFINITY;
    for (int64_t v = 0; v < V; ++v) {
        const double raw = (double)logits[v];
        if (isnan(raw) || (isinf(raw) && raw > 0)) return 1;
        const double l = raw / T;
        if (l > m) m = l;
    }
    if (isinf(m)) return 1;
    double z = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        prob[v] = exp((double)logits[v] / T - m);
        z += prob[v];
    }
    for (int64_t v = 0; v < V; ++v) prob[v] /= z;
    return 0;
}

/* Inverse CDF with one uniform u in [0,1): the smallest v whose cumulative
 * weight C(v) = w[0] + ... + w[v] exceeds u * S, S = C(V-1); the vocabulary
 * order is the order of the CDF.  *margin receives the distance from u*S to
 * the nearer edge of the chosen bucket, relative to S. */
static int32_t inv_cdf_f64(const double *w, double u, int64_t V, double *margin)
{
    double S = 0.0;
    for (int64_t v = 0; v < V; ++v) S += w[v];
    const double t = u * S;
    double c = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        const double prev = c;
        c += w[v];
        if (c > t) {
            if (margin) *margin = fmin(c - t, t - prev) / S;
            return (int32_t)v;
        }
    }
    for (int64_t v = V - 1; v >= 0; --v)
        if (w[v] > 0.0) {
            if (margin) *margin = 0.0;
            return (int32_t)v;
        }
    return -1;
}

/* As oracle_verify_block_f64, at temperature T > 0, with the resample drawn
 * by mode 0 (exponential race, u_res [Bn,V]) or mode 1 (inverse CDF, u_res
 * [Bn], one uniform in [0,1) per sequence).  race_margin receives the race's
 * margin or, in mode 1, the inverse CDF's. */
int oracle_verify_block_ex_f64(const float *p_logits, const float *q_logits,
                               const int32_t *draft, const float *u_acc,
                               const float *u_res, int64_t Bn, int64_t K,
                               int64_t Kp, int64_t V, double T, int mode,
                               int32_t *n_accepted, int32_t *out_tokens,
                               int32_t *n_emitted, int32_t *status,
                               double *accept_margin, double *race_margin)
{
    if (Bn < 0 || K < 0 || V <= 0 || (Kp != K && Kp != K + 1)) return OR_ERR_ARG;
    if (!(T > 0.0) || isinf(T) || (mode != 0 && mode != 1)) return OR_ERR_ARG;
    if (Bn == 0) return OR_OK;
    if (!p_logits || (K > 0 && (!q_logits || !draft || !u_acc)) || !u_res ||
        !n_accepted || !out_tokens || !n_emitted || !status)
        return OR_ERR_ARG;
    int err = OR_OK;

#pragma omp parallel
    {
        double *P = (double *)malloc(sizeof(double) * (size_t)(Kp > 0 ? Kp : 1) * (size_t)V);
        double *Q = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1) * (size_t)V);
        double *r = (double *)malloc(sizeof(double) * (size_t)V);
        if (!P || !Q || !r) {
#pragma omp atomic write
            err = OR_ERR_NOMEM;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t b = 0; b < Bn; ++b) {
            if (!P || !Q || !r) continue;
            int32_t *out = out_tokens + b * (K + 1);
            for (int64_t i = 0; i <= K; ++i) out[i] = -1;
            if (accept_margin)
                for (int64_t i = 0; i < K; ++i) accept_margin[b * K + i] = INFINITY;
            if (race_margin) race_margin[b] = INFINITY;
            n_accepted[b] = 0;
            n_emitted[b] = 0;
            status[b] = OR_SEQ_OK;

            for (int64_t i = 0; i < K; ++i) {
                const int32_t x = draft[b * K + i];
                if (x < 0 || x >= V) status[b] = OR_SEQ_BAD_DRAFT;
            }
            /* Step 1: softmax of every row at temperature T. */
            int bad = 0;
            for (int64_t i = 0; i < Kp; ++i)
                bad |= softmax_row_temp_f64(p_logits + (b * Kp + i) * V, V, T, P + i * V);
            for (int64_t i = 0; i < K; ++i)
                bad |= softmax_row_temp_f64(q_logits + (b * K + i) * V, V, T, Q + i * V);
            if (bad && status[b] == OR_SEQ_OK) status[b] = OR_SEQ_NONFINITE;
            if (status[b] != OR_SEQ_OK) continue;

            /* Step 2: the acceptance rule, unchanged. */
            int64_t n = 0;
            for (int64_t i = 0; i < K; ++i) {
                const int32_t x = draft[b * K + i];
                const double pi = P[i * V + x];
                const double qi = Q[i * V + x];
                const double rho = qi > 0.0 ? pi / qi : INFINITY;
                const double thr = rho < 1.0 ? rho : 1.0;
                const double u = (double)u_acc[b * K + i];
                if (accept_margin) accept_margin[b * K + i] = fabs(thr - u);
                if (u < thr) {
                    out[i] = x;
                    ++n;
                } else {
                    break;
                }
            }
            n_accepted[b] = (int32_t)n;
            n_emitted[b] = (int32_t)n;

            /* Step 3: the residual (or bonus) token, by the chosen sampler. */
            double *rm = race_margin ? race_margin + b : NULL;
            const double *w = NULL;
            if (n < K) {
                double S = 0.0;
                for (int64_t v = 0; v < V; ++v) {
                    const double d = P[n * V + v] - Q[n * V + v];
                    r[v] = d > 0.0 ? d : 0.0;
                    S += r[v];
                }
                if (S == 0.0)
                    for (int64_t v = 0; v < V; ++v) r[v] = P[n * V + v];
                w = r;
            } else if (Kp == K + 1) {
                w = P + K * V;
            }
            if (w) {
                out[n] = mode == 0 ? race_f64(w, u_res + b * V, V, rm)
                                   : inv_cdf_f64(w, (double)u_res[b], V, rm);
                n_emitted[b] = (int32_t)(n + 1);
            }
        }
        free(P);
        free(Q);
        free(r);
    }
    return err;
}

/* ------------------------------------------------------------------------ */
/* LM head feeding the verifier.  [Explainer] "The Psi-Spec Sampler": the   */
/* AR model verifies the drafted block in a single forward pass; its last   */
/* step is the LM head, logits = h . W^T over the vocabulary, for the AR    */
/* rows (h_p [Bn,Kp,d], head W_p [V,d]) and the draft rows (h_q [Bn,K,d],   */
/* head W_q [V,d]; the same matrix when both pathways share the head).      */
/* The result is the verifier's on those logits, computed here in fp64     */
/* from the fp64 dot products (no rounding of the logits).                  */
/* ------------------------------------------------------------------------ */
static int softmax_dlogits_f64(const double *l, int64_t V, double *prob)
{
    double m = -INFINITY;
    for (int64_t v = 0; v < V; ++v) {
        if (isnan(l[v]) || (isinf(l[v]) && l[v] > 0)) return 1;
        if (l[v] > m) m = l[v];
    }
    if (isinf(m)) return 1;
    double z = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        prob[v] = exp(l[v] - m);
        z += prob[v];
    }
    for (int64_t v = 0; v < V; ++v) prob[v] /= z;
    return 0;
}

/* logits[v] = sum_k h[k] * W[v, k] */
static void lm_head_row_f64(const double *h, const double *W, int64_t d, int64_t V, double *logits)
{
    for (int64_t v = 0; v < V; ++v) {
        double acc = 0.0;
        for (int64_t k = 0; k < d; ++k) acc += h[k] * W[v * d + k];
        logits[v] = acc;
    }
}

int oracle_lm_head_verify_f64(const double *h_p, const double *h_q, const double *W_p,
                              const double *W_q, int64_t d, const int32_t *draft,
                              const float *u_acc, const float *u_res, int64_t Bn, int64_t K,
                              int64_t Kp, int64_t V, int32_t *n_accepted, int32_t *out_tokens,
                              int32_t *n_emitted, int32_t *status, double *accept_margin,
                              double *race_margin)
{
    if (Bn < 0 || K < 0 || V <= 0 || d <= 0 || (Kp != K && Kp != K + 1)) return OR_ERR_ARG;
    if (Bn == 0) return OR_OK;
    if (!h_p || !W_p || (K > 0 && (!h_q || !W_q || !draft || !u_acc)) || !u_res ||
        !n_accepted || !out_tokens || !n_emitted || !status)
        return OR_ERR_ARG;
    int err = OR_OK;

#pragma omp parallel
    {
        double *P = (double *)malloc(sizeof(double) * (size_t)(Kp > 0 ? Kp : 1) * (size_t)V);
        double *Q = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1) * (size_t)V);
        double *l = (double *)malloc(sizeof(double) * (size_t)V);
        double *r = (double *)malloc(sizeof(double) * (size_t)V);
        if (!P || !Q || !l || !r) {
#pragma omp atomic write
            err = OR_ERR_NOMEM;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t b = 0; b < Bn; ++b) {
            if (!P || !Q || !l || !r) continue;
            int32_t *out = out_tokens + b * (K + 1);
            for (int64_t i = 0; i <= K; ++i) out[i] = -1;
            if (accept_margin)
                for (int64_t i = 0; i < K; ++i) accept_margin[b * K + i] = INFINITY;
            if (race_margin) race_margin[b] = INFINITY;
            n_accepted[b] = 0;
            n_emitted[b] = 0;
            status[b] = OR_SEQ_OK;
            for (int64_t i = 0; i < K; ++i) {
                const int32_t x = draft[b * K + i];
                if (x < 0 || x >= V) status[b] = OR_SEQ_BAD_DRAFT;
            }
            /* Step 1: the LM head, then the softmax of every row. */
            int bad = 0;
            for (int64_t i = 0; i < Kp; ++i) {
                lm_head_row_f64(h_p + (b * Kp + i) * d, W_p, d, V, l);
                bad |= softmax_dlogits_f64(l, V, P + i * V);
            }
            for (int64_t i = 0; i < K; ++i) {
                lm_head_row_f64(h_q + (b * K + i) * d, W_q, d, V, l);
                bad |= softmax_dlogits_f64(l, V, Q + i * V);
            }
            if (bad && status[b] == OR_SEQ_OK) status[b] = OR_SEQ_NONFINITE;
            if (status[b] != OR_SEQ_OK) continue;
            /* Step 2: accept x_i iff u_i < min(1, p_i(x_i)/q_i(x_i)). */
            int64_t n = 0;
            for (int64_t i = 0; i < K; ++i) {
                const int32_t x = draft[b * K + i];
                const double pi = P[i * V + x];
                const double qi = Q[i * V + x];
                const double rho = qi > 0.0 ? pi / qi : INFINITY;
                const double thr = rho < 1.0 ? rho : 1.0;
                const double u = (double)u_acc[b * K + i];
                if (accept_margin) accept_margin[b * K + i] = fabs(thr - u);
                if (u < thr) {
                    out[i] = x;
                    ++n;
                } else {
                    break;
                }
            }
            n_accepted[b] = (int32_t)n;
            n_emitted[b] = (int32_t)n;
            /* Step 3: the residual or bonus token by the exponential race. */
            const float *ub = u_res + b * V;
            double *rm = race_margin ? race_margin + b : NULL;
            if (n < K) {
                double S = 0.0;
                for (int64_t v = 0; v < V; ++v) {
                    const double dd = P[n * V + v] - Q[n * V + v];
                    r[v] = dd > 0.0 ? dd : 0.0;
                    S += r[v];
                }
                if (S == 0.0)
                    for (int64_t v = 0; v < V; ++v) r[v] = P[n * V + v];
                out[n] = race_f64(r, ub, V, rm);
                n_emitted[b] = (int32_t)(n + 1);
            } else if (Kp == K + 1) {
                out[K] = race_f64(P + K * V, ub, V, rm);
                n_emitted[b] = (int32_t)(K + 1);
            }
        }
        free(P);
        free(Q);
        free(l);
        free(r);
    }
    return err;
}

/* ------------------------------------------------------------------------ */
/* Tree sampler, verification half.  [Explainer] "The Psi-Spec Sampler":    */
/* the tree sampler takes several candidates (the top K) at each position   */
/* and verifies them in a prefix tree, keeping the AR model's distribution. */
/* Each drafted node is a deterministic candidate, i.e. a point-mass draft  */
/* q = delta_x, for which the speculative rule reads: accept x with         */
/* probability r(x)/S (r the current residual, S its mass), else remove x   */
/* from the residual, max(0, r - delta_x), and try the next candidate.      */
/* Walking down from the root: at the current node test its children in     */
/* index order (their rank); on an acceptance emit the child's token and    */
/* move to it; when every child is rejected (or there are none) draw one    */
/* token from the residual by the exponential race and stop.                */
/*                                                                          */
/* logits [Bn, N+1, V]: AR logits for the token after node j (node 0 is the */
/* committed prefix); parent [Bn, N+1] with parent[0] = -1 and              */
/* 0 <= parent[j] < j; token [Bn, N+1] (token[0] unused); u_acc [Bn, N+1]   */
/* (the test of node j uses u_acc[j]); u_res [Bn, V].  Outputs n_accepted   */
/* [Bn] (accepted depth), path [Bn, N] accepted node ids (-1 padded),       */
/* out_tokens [Bn, N+1] (-1 padded), n_emitted [Bn], status [Bn]; optional  */
/* accept_margin [Bn, N+1] |r(x)/S - u| per tested node, race_margin [Bn].  */
/* ------------------------------------------------------------------------ */
int oracle_tree_verify_f64(const float *logits, const int32_t *parent, const int32_t *token,
                           const float *u_acc, const float *u_res, int64_t Bn, int64_t N,
                           int64_t V, int32_t *n_accepted, int32_t *path, int32_t *out_tokens,
                           int32_t *n_emitted, int32_t *status, double *accept_margin,
                           double *race_margin)
{
    if (Bn < 0 || N < 0 || V <= 0) return OR_ERR_ARG;
    if (Bn == 0) return OR_OK;
    if (!logits || !parent || !token || !u_acc || !u_res || !n_accepted || !path ||
        !out_tokens || !n_emitted || !status)
        return OR_ERR_ARG;
    int err = OR_OK;

#pragma omp parallel
    {
        double *r = (double *)malloc(sizeof(double) * (size_t)V);
        if (!r) {
#pragma omp atomic write
            err = OR_ERR_NOMEM;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t b = 0; b < Bn; ++b) {
            if (!r) continue;
            const int32_t *par = parent + b * (N + 1);
            const int32_t *tok = token + b * (N + 1);
            int32_t *out = out_tokens + b * (N + 1);
            int32_t *pth = path + b * N;
            for (int64_t i = 0; i <= N; ++i) out[i] = -1;
            for (int64_t i = 0; i < N; ++i) pth[i] = -1;
            if (accept_margin)
                for (int64_t i = 0; i <= N; ++i) accept_margin[b * (N + 1) + i] = INFINITY;
            if (race_margin) race_margin[b] = INFINITY;
            n_accepted[b] = 0;
            n_emitted[b] = 0;
            status[b] = OR_SEQ_OK;
            /* a tree in topological order with tokens inside the vocabulary */
            int ok = par[0] == -1;
            for (int64_t j = 1; j <= N; ++j)
                ok &= par[j] >= 0 && par[j] < j && tok[j] >= 0 && tok[j] < V;
            if (!ok) {
                status[b] = OR_SEQ_BAD_DRAFT;
                continue;
            }
            int64_t cur = 0, depth = 0;
            while (1) {
                if (softmax_row_f64(logits + (b * (N + 1) + cur) * V, V, r)) {
                    status[b] = OR_SEQ_NONFINITE;
                    break;
                }
                double S = 1.0;
                int64_t acc = -1;
                for (int64_t j = cur + 1; j <= N && acc < 0; ++j) {
                    if (par[j] != cur) continue;
                    const int32_t x = tok[j];
                    const double thr = S > 0.0 ? r[x] / S : 0.0;
                    const double u = (double)u_acc[b * (N + 1) + j];
                    if (accept_margin) accept_margin[b * (N + 1) + j] = fabs(thr - u);
                    if (u < thr) {
                        acc = j;
                    } else {
                        S -= r[x];
                        r[x] = 0.0;
                    }
                }
                if (acc >= 0) {
                    out[depth] = tok[acc];
                    pth[depth] = (int32_t)acc;
                    ++depth;
                    cur = acc;
                    continue;
                }
                /* every child rejected: one token from the residual (from
                 * p itself should rounding have emptied the residual) */
                double mass = 0.0;
                for (int64_t v = 0; v < V; ++v) mass += r[v];
                if (!(mass > 0.0)) softmax_row_f64(logits + (b * (N + 1) + cur) * V, V, r);
                out[depth] = race_f64(r, u_res + b * V, V, race_margin ? race_margin + b : NULL);
                break;
            }
            if (status[b] != OR_SEQ_OK) {
                for (int64_t i = 0; i <= N; ++i) out[i] = -1;
                for (int64_t i = 0; i < N; ++i) pth[i] = -1;
                continue;
            }
            n_accepted[b] = (int32_t)depth;
            n_emitted[b] = (int32_t)(depth + 1);
        }
        free(r);
    }
    return err;
}

/* ------------------------------------------------------------------------ */
/* Draft sampling (Psi-Spec linear sampler, drafting half).                 */
/* [Explainer] "The Psi-Spec Sampler": the linear sampler draws one         */
/* candidate per token position.  tokens[r] = argmax_v q_r(v) / (-ln u[r,v])*/
/* with q_r = softmax(logits[r,:]); status[r] = 2 for a non-finite row.     */
/* ------------------------------------------------------------------------ */
int oracle_draft_sample_f64(const float *logits, const float *u, int64_t R,
                            int64_t V, int32_t *tokens, int32_t *status,
                            double *margin)
{
    if (R < 0 || V <= 0) return OR_ERR_ARG;
    if (R == 0) return OR_OK;
    if (!logits || !u || !tokens || !status) return OR_ERR_ARG;
    int err = OR_OK;
#pragma omp parallel
    {
        double *q = (double *)malloc(sizeof(double) * (size_t)V);
        if (!q) {
#pragma omp atomic write
            err = OR_ERR_NOMEM;
        }
#pragma omp for schedule(dynamic, 4)
        for (int64_t row = 0; row < R; ++row) {
            if (!q) continue;
            if (softmax_row_f64(logits + row * V, V, q)) {
                tokens[row] = -1;
                status[row] = OR_SEQ_NONFINITE;
                if (margin) margin[row] = INFINITY;
                continue;
            }
            status[row] = OR_SEQ_OK;
            tokens[row] = race_f64(q, u + row * V, V, margin ? margin + row : NULL);
        }
        free(q);
    }
    return err;
}

/* Number of host threads the oracle's parallel regions use. */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
