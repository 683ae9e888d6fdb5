/*
 * kda_oracle.c -- float64 CPU oracle for the Kimi Delta Attention (KDA)
 * state recurrence.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check and
 * the bench's CPU-baseline / reference legs may load this library.  It shares
 * no code, header, table or helper with the CUDA library, and it never calls
 * into it.
 *
 * What it computes (the plain definition, one token at a time, in float64):
 *
 *   Source: "[논문 리뷰] Kimi K3 Technical Report" (jw9603.github.io),
 *   section 3.2 (state update and readout), section 3.3 (delta-rule form),
 *   section 3.5 (alpha = exp(g)).
 *
 *     alpha_t   = exp(g_t)                         (sec. 3.5; g = log_alpha)
 *     Sbar      = Diag(alpha_t) S_{t-1}            (sec. 3.3; row i of S is
 *                                                   key channel i, scaled by
 *                                                   alpha_t[i], sec. 3.2)
 *     S_t       = Sbar + beta_t k_t (v_t - Sbar^T k_t)^T       (sec. 3.3)
 *               = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1}
 *                 + beta_t k_t v_t^T                            (sec. 3.2)
 *     o_t       = S_t^T q_t      (sec. 3.2: read with the state that already
 *                                 holds token t's write)
 *
 * Shapes and layouts (all row-major, all float64):
 *   q, k, log_alpha : [T_tot, H, dk]
 *   v, o            : [T_tot, H, dv]
 *   beta            : [T_tot, H]
 *   S0, S_final     : [N, H, dk, dv]   (row index = key channel)
 *   cu_seqlens      : [N + 1], cu[0] = 0, non-decreasing, cu[N] = T_tot;
 *                     sequence n owns tokens cu[n] .. cu[n+1]-1.
 *
 * Nothing here assumes beta in (0,1) or a unit-norm k; the update is applied
 * exactly as written for any finite inputs.  No clamping of g is done.
 *
 * Independent (sequence, head) units run on a small pthread pool; each unit is
 * processed by exactly one thread in token order, so the result does not
 * depend on the thread count.
 *
 * Parity pins (tests/test_oracle_pins.py): the section-3.4 worked example,
 * beta/alpha special cases, the section-3.2 diagonal example, the explicit
 * product form of section 3.2, the gradient-step reading of the delta rule,
 * the Householder reflection at beta = 2, closed forms for a repeated key and
 * for orthonormal keys, and a brute-force dense-matrix unrolling on tiny cases.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const double *q, *k, *v, *log_alpha, *beta, *S0;
    const int64_t *cu_seqlens;
    int64_t num_seqs, H, dk, dv;
    double *o, *S_final;
    int nthreads;
    int tid;
} oracle_job;

/* One (sequence n, head h) unit: run the recurrence over the sequence's
 * tokens, writing o for each token and the final state. */
static void run_unit(const oracle_job *J, int64_t n, int64_t h, double *S,
                     double *alpha, double *err)
{
    const int64_t H = J->H, dk = J->dk, dv = J->dv;
    const int64_t state_off = (n * H + h) * dk * dv;

    if (J->S0) {
        memcpy(S, J->S0 + state_off, (size_t)(dk * dv) * sizeof(double));
    } else {
        memset(S, 0, (size_t)(dk * dv) * sizeof(double));
    }

    for (int64_t t = J->cu_seqlens[n]; t < J->cu_seqlens[n + 1]; ++t) {
        const double *qt = J->q + (t * H + h) * dk;
        const double *kt = J->k + (t * H + h) * dk;
        const double *gt = J->log_alpha + (t * H + h) * dk;
        const double *vt = J->v + (t * H + h) * dv;
        const double bt = J->beta[t * H + h];
        double *ot = J->o + (t * H + h) * dv;

        /* alpha_t = exp(g_t), per key channel. */
        for (int64_t i = 0; i < dk; ++i) alpha[i] = exp(gt[i]);

        /* Sbar = Diag(alpha_t) S_{t-1}: scale row i by alpha_t[i]. */
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j) S[i * dv + j] *= alpha[i];

        /* err = v_t - Sbar^T k_t  (the value the memory gets wrong). */
        for (int64_t j = 0; j < dv; ++j) {
            double pred = 0.0;
            for (int64_t i = 0; i < dk; ++i) pred += S[i * dv + j] * kt[i];
            err[j] = vt[j] - pred;
        }

        /* S_t = Sbar + beta_t k_t err^T. */
        for (int64_t i = 0; i < dk; ++i) {
            const double bk = bt * kt[i];
            for (int64_t j = 0; j < dv; ++j) S[i * dv + j] += bk * err[j];
        }

        /* o_t = S_t^T q_t. */
        for (int64_t j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int64_t i = 0; i < dk; ++i) acc += S[i * dv + j] * qt[i];
            ot[j] = acc;
        }
    }

    if (J->S_final)
        memcpy(J->S_final + state_off, S, (size_t)(dk * dv) * sizeof(double));
}

static void *worker(void *arg)
{
    const oracle_job *J = (const oracle_job *)arg;
    const int64_t units = J->num_seqs * J->H;
    double *S = (double *)malloc((size_t)(J->dk * J->dv) * sizeof(double));
    double *alpha = (double *)malloc((size_t)J->dk * sizeof(double));
    double *err = (double *)malloc((size_t)J->dv * sizeof(double));
    if (S && alpha && err) {
        for (int64_t u = J->tid; u < units; u += J->nthreads)
            run_unit(J, u / J->H, u % J->H, S, alpha, err);
    }
    free(S);
    free(alpha);
    free(err);
    return NULL;
}

/* Returns 0 on success, 1 on an invalid argument, 2 if a thread could not be
 * started.  o must hold T_tot*H*dv doubles; S_final may be NULL. */
int kda_oracle_prefill(const double *q, const double *k, const double *v,
                       const double *log_alpha, const double *beta,
                       const double *S0, const int64_t *cu_seqlens,
                       int64_t num_seqs, int64_t H, int64_t dk, int64_t dv,
                       double *o, double *S_final, int nthreads)
{
    if (!q || !k || !v || !log_alpha || !beta || !cu_seqlens || !o) return 1;
    if (num_seqs < 1 || H < 1 || dk < 1 || dv < 1) return 1;
    if (cu_seqlens[0] != 0) return 1;
    for (int64_t n = 0; n < num_seqs; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return 1;

    int64_t units = num_seqs * H;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > units) nthreads = (int)units;
    if (nthreads > 256) nthreads = 256;

    oracle_job jobs[256];
    pthread_t th[256];
    for (int i = 0; i < nthreads; ++i) {
        oracle_job J = {q, k, v, log_alpha, beta, S0, cu_seqlens, num_seqs,
                        H, dk, dv, o, S_final, nthreads, i};
        jobs[i] = J;
    }
    int started = 0, rc = 0;
    for (int i = 1; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, worker, &jobs[i]) != 0) {
            rc = 2;
            break;
        }
        started = i;
    }
    if (rc == 0) worker(&jobs[0]);
    for (int i = 1; i <= started; ++i) pthread_join(th[i], NULL);
    return rc;
}

/* One decode step for N independent sequences: the recurrence above applied
 * to a single token per (sequence, head), state updated in place.
 * q, k, log_alpha: [N, H, dk]; v, o: [N, H, dv]; beta: [N, H];
 * S_inout: [N, H, dk, dv]. */
int kda_oracle_decode_step(const double *q, const double *k, const double *v,
                           const double *log_alpha, const double *beta,
                           double *S_inout, int64_t N, int64_t H, int64_t dk,
                           int64_t dv, double *o, int nthreads)
{
    if (N < 1) return 1;
    int64_t *cu = (int64_t *)malloc((size_t)(N + 1) * sizeof(int64_t));
    if (!cu) return 2;
    for (int64_t n = 0; n <= N; ++n) cu[n] = n;
    int rc = kda_oracle_prefill(q, k, v, log_alpha, beta, S_inout, cu, N, H,
                                dk, dv, o, S_inout, nthreads);
    free(cu);
    return rc;
}
