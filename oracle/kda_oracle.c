/*
 * KDA (Kimi Delta Attention) forward -- plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the test-suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header or constant with the CUDA
 * library.
 *
 * What it computes (per sequence n and head h, independently):
 *
 *     S_0 = initial state (d_k x d_v, zero when none is given)
 *     for t = 1..T:
 *         S'  = Diag(exp(log_alpha_t)) . S_{t-1}     row c scaled by alpha_tc
 *         u   = beta_t * (v_t - S'^T k_t)             a d_v vector
 *         S_t = S' + k_t u^T                          the delta-rule write
 *         o_t = scale * S_t^T q_t
 *
 * which is S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T,
 * the gated delta rule with one decay per key channel.  The pages describe
 * it in words: orkas.ai "Kimi K3 architecture" (German edition), section
 * "Sequenz: Drei Viertel der Schichten lesen nicht mehr alles" (a running
 * state of fixed size; a decay that makes recent tokens more present) and
 * section "Die Rechnung landet in der Bereitstellungsinfrastruktur" (the
 * state is updated serially and in place).  Decay first, then the delta
 * rule on the decayed state, and the output reads the updated state.
 *
 * Columns of S evolve independently (the transition acts from the left), so
 * the work is split over (head, block of d_v columns) with OpenMP.
 *
 * Layouts (all row-major, fp64):
 *   q, k, log_alpha : [T_total][H][d_k]
 *   v               : [T_total][H][d_v]
 *   beta            : [T_total][H]
 *   cu_seqlens      : [N+1]  (sequence n owns tokens cu[n] .. cu[n+1]-1)
 *   initial_state   : [N][H][d_k][d_v] or NULL (zeros)
 *   out             : [T_total][H][d_v]
 *   final_state     : [N][H][d_k][d_v] or NULL (not written)
 *
 * `mutation` plants a known mistake for the tests that prove the pins have
 * teeth (0 = the method as defined).  See kda_oracle.h.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#include "kda_oracle.h"

#define COLS_PER_TASK 8

int kda_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static void run_task(int n, int h, int j0, int j1, int H, int dk, int dv,
                     const long long* cu, const double* q, const double* k,
                     const double* v, const double* log_alpha,
                     const double* beta, const double* initial_state,
                     double scale, double* out, double* final_state,
                     int mutation, double* S /* [dk][COLS] scratch */,
                     double* alpha /* [dk] */) {
    const int nc = j1 - j0;
    const long long t_begin = cu[n], t_end = cu[n + 1];
    /* S[c*COLS + jj] holds state entry (c, j0+jj). */
    for (int c = 0; c < dk; ++c)
        for (int jj = 0; jj < nc; ++jj)
            S[c * COLS_PER_TASK + jj] =
                initial_state
                    ? initial_state[(((long long)n * H + h) * dk + c) * dv + j0 + jj]
                    : 0.0;

    for (long long t = t_begin; t < t_end; ++t) {
        const double* qt = q + (t * H + h) * dk;
        const double* kt = k + (t * H + h) * dk;
        const double* vt = v + (t * H + h) * dv;
        const double* lat = log_alpha + (t * H + h) * dk;
        const double bt = beta[t * H + h];
        for (int c = 0; c < dk; ++c) alpha[c] = exp(lat[c]);

        for (int jj = 0; jj < nc; ++jj) {
            const int j = j0 + jj;
            double kS = 0.0;
            if (mutation == KDA_MUT_DECAY_AFTER_WRITE) {
                /* wrong order: write on the undecayed state, decay after */
                for (int c = 0; c < dk; ++c) kS += S[c * COLS_PER_TASK + jj] * kt[c];
                const double u = bt * (vt[j] - kS);
                for (int c = 0; c < dk; ++c) {
                    double s = S[c * COLS_PER_TASK + jj] + kt[c] * u;
                    S[c * COLS_PER_TASK + jj] = alpha[c] * s;
                }
            } else {
                /* S' = Diag(alpha) S ; kS = S'^T k */
                for (int c = 0; c < dk; ++c) {
                    double s = S[c * COLS_PER_TASK + jj];
                    if (mutation == KDA_MUT_DECAY_ON_COLUMNS)
                        s *= exp(lat[j % dk]);
                    else
                        s *= alpha[c];
                    S[c * COLS_PER_TASK + jj] = s;
                    kS += s * kt[c];
                }
                double u;
                if (mutation == KDA_MUT_DROP_BETA)
                    u = vt[j] - kS;
                else if (mutation == KDA_MUT_SIGN)
                    u = bt * (vt[j] + kS);
                else
                    u = bt * (vt[j] - kS);
                if (mutation == KDA_MUT_OUTPUT_BEFORE_WRITE) {
                    double o = 0.0;
                    for (int c = 0; c < dk; ++c) o += S[c * COLS_PER_TASK + jj] * qt[c];
                    out[(t * H + h) * dv + j] = scale * o;
                    for (int c = 0; c < dk; ++c) S[c * COLS_PER_TASK + jj] += kt[c] * u;
                    continue;
                }
                for (int c = 0; c < dk; ++c) S[c * COLS_PER_TASK + jj] += kt[c] * u;
            }
            double o = 0.0;
            for (int c = 0; c < dk; ++c) o += S[c * COLS_PER_TASK + jj] * qt[c];
            out[(t * H + h) * dv + j] = scale * o;
        }
    }
    if (final_state)
        for (int c = 0; c < dk; ++c)
            for (int jj = 0; jj < nc; ++jj)
                final_state[(((long long)n * H + h) * dk + c) * dv + j0 + jj] =
                    S[c * COLS_PER_TASK + jj];
}

int kda_oracle_fwd(int N, int H, int dk, int dv, const long long* cu_seqlens,
                   const double* q, const double* k, const double* v,
                   const double* log_alpha, const double* beta,
                   const double* initial_state, double scale, double* out,
                   double* final_state, int num_threads, int mutation) {
    if (N < 0 || H <= 0 || dk <= 0 || dv <= 0 || !cu_seqlens) return 1;
    for (int n = 0; n < N; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return 1;
    if (mutation == KDA_MUT_DECAY_ON_COLUMNS && dk != dv) return 1;
    const int blocks = (dv + COLS_PER_TASK - 1) / COLS_PER_TASK;
    const long long tasks = (long long)N * H * blocks;
    int err = 0;
#ifdef _OPENMP
    if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel num_threads(num_threads)
#endif
    {
        double* S = (double*)malloc(sizeof(double) * (size_t)dk * COLS_PER_TASK);
        double* alpha = (double*)malloc(sizeof(double) * (size_t)dk);
        if (!S || !alpha) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            err = 2;
        } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
            for (long long task = 0; task < tasks; ++task) {
                const int b = (int)(task % blocks);
                const int h = (int)((task / blocks) % H);
                const int n = (int)(task / ((long long)blocks * H));
                const int j0 = b * COLS_PER_TASK;
                const int j1 = j0 + COLS_PER_TASK < dv ? j0 + COLS_PER_TASK : dv;
                run_task(n, h, j0, j1, H, dk, dv, cu_seqlens, q, k, v, log_alpha, beta,
                         initial_state, scale, out, final_state, mutation, S, alpha);
            }
        }
        free(S);
        free(alpha);
    }
    return err;
}
