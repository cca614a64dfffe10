/*
 * KDA oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, token-by-token CPU evaluation of the Kimi Delta Attention
 * (KDA) forward recurrence in double precision.  Only the test suite, the
 * smoke check and the CPU-baseline leg of the benchmark may load this file's
 * library; the product path never does.  It shares no code, header or
 * constant with the CUDA library.
 *
 * What it computes (one independent chain per (sequence n, head h)):
 *
 *   S = h0[n,h]  (dk x dv, or zeros)
 *   for each token t of sequence n, in order:
 *       S   <- diag(exp(g_t)) S                  channel-wise forget gate
 *       S   <- S + beta_t k_t (v_t - S^T k_t)^T  delta-rule write
 *       o_t  = scale * S^T q_t                   read-out from the updated S
 *   hT[n,h] = S
 *
 * Sources: "Kimi K3 技术报告摘要" (gkm0120.cn/p/60370.html), section 1
 * 预训练 Recipe, 训练策略 table, KDA row: delta-rule recurrence with a
 * channel-wise forget gate.  "Kimi K3 NPU Training", section 模型结构
 * (KDA gives each channel its own forget gate, q/k are L2-normalised,
 * decode keeps one fixed matrix state per head) and section 定长与 TND
 * (the recurrent state resets at every packed-sequence boundary).
 * The tensor g carries log(alpha) directly (natural log, g <= 0).
 *
 * Layout: token-major packed activations x[(t*H + h)*d + c] for the global
 * token index t; sequence n owns tokens [cu[n], cu[n+1]).  States are
 * [N, H, dk, dv] with dv fastest.  Inputs are float or double arrays (every
 * bf16 and fp32 value is exact in either) and are widened to double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Element i of an input array that holds floats (f64 == 0) or doubles. */
static inline double ld(const void *p, int64_t i, int f64)
{
    return f64 ? ((const double *)p)[i] : (double)((const float *)p)[i];
}

/* Evaluate one (sequence, head) chain.  Returns 0, or -1 on allocation failure. */
static int kda_chain(int64_t t0, int64_t t1, int64_t h, int64_t H, int64_t dk, int64_t dv,
                     const void *q, const void *k, const void *v, const void *g,
                     const void *beta, const void *h0, int64_t h0_off, int f64,
                     double scale, double *o, double *hT_nh)
{
    double *S = (double *)malloc(sizeof(double) * (size_t)(dk * dv));
    double *a = (double *)malloc(sizeof(double) * (size_t)dk);
    double *kt = (double *)malloc(sizeof(double) * (size_t)dk);
    double *p = (double *)malloc(sizeof(double) * (size_t)dv);
    if (!S || !a || !kt || !p) { free(S); free(a); free(kt); free(p); return -1; }

    for (int64_t i = 0; i < dk * dv; ++i) S[i] = h0 ? ld(h0, h0_off + i, f64) : 0.0;

    for (int64_t t = t0; t < t1; ++t) {
        const int64_t xk = (t * H + h) * dk, xv = (t * H + h) * dv;
        const double bt = ld(beta, t * H + h, f64);

        /* decay: S <- diag(alpha_t) S, alpha_t = exp(g_t) per key channel */
        for (int64_t i = 0; i < dk; ++i) a[i] = exp(ld(g, xk + i, f64));
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j) S[i * dv + j] *= a[i];

        /* prediction p = S^T k_t from the decayed state */
        for (int64_t i = 0; i < dk; ++i) kt[i] = ld(k, xk + i, f64);
        for (int64_t j = 0; j < dv; ++j) p[j] = 0.0;
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j) p[j] += S[i * dv + j] * kt[i];

        /* delta write: S <- S + beta_t k_t (v_t - p)^T */
        for (int64_t j = 0; j < dv; ++j) p[j] = bt * (ld(v, xv + j, f64) - p[j]);
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j) S[i * dv + j] += kt[i] * p[j];

        /* read-out from the updated state: o_t = scale * S^T q_t */
        if (o) {
            double *ot = o + xv;
            for (int64_t j = 0; j < dv; ++j) ot[j] = 0.0;
            for (int64_t i = 0; i < dk; ++i) {
                const double qi = ld(q, xk + i, f64);
                for (int64_t j = 0; j < dv; ++j) ot[j] += S[i * dv + j] * qi;
            }
            for (int64_t j = 0; j < dv; ++j) ot[j] *= scale;
        }
    }
    if (hT_nh) memcpy(hT_nh, S, sizeof(double) * (size_t)(dk * dv));
    free(S); free(a); free(kt); free(p);
    return 0;
}

/*
 * Run every (sequence, head) chain.  cu has n_seqs+1 entries (token offsets,
 * non-decreasing).  f64 selects double (1) or float (0) for every input array
 * (q, k, v, g, beta, h0).  h0 may be NULL (zero start state); o and hT may be
 * NULL.  Chains are independent, so they are spread over n_threads OpenMP
 * threads; the arithmetic inside a chain is exactly the loop above.
 * Returns 0 on success, -1 on bad arguments or allocation failure.
 */
int kda_oracle_recurrent(int64_t n_seqs, const int64_t *cu, int64_t H, int64_t dk, int64_t dv,
                         const void *q, const void *k, const void *v, const void *g,
                         const void *beta, const void *h0, int f64, double scale,
                         double *o, double *hT, int n_threads)
{
    if (n_seqs < 0 || H <= 0 || dk <= 0 || dv <= 0 || !cu) return -1;
    for (int64_t n = 0; n < n_seqs; ++n)
        if (cu[n + 1] < cu[n]) return -1;
    const int64_t chains = n_seqs * H;
    int err = 0;
    if (n_threads < 1) n_threads = 1;
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads) reduction(| : err)
    for (int64_t c = 0; c < chains; ++c) {
        const int64_t n = c / H, h = c % H;
        const int64_t st = (n * H + h) * dk * dv;
        err |= kda_chain(cu[n], cu[n + 1], h, H, dk, dv, q, k, v, g, beta, h0, st, f64,
                         scale, o, hT ? hT + st : NULL) != 0;
    }
    return err ? -1 : 0;
}

/* Number of threads OpenMP would use by default (the host's usable cores). */
int kda_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
