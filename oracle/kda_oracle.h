/*
 * fp64 CPU oracle of the KDA forward recurrence -- TEST INFRASTRUCTURE ONLY.
 * Shares nothing with the CUDA library; see kda_oracle.c for the definition.
 */
#ifndef KDA_ORACLE_H
#define KDA_ORACLE_H

#ifdef __cplusplus
extern "C" {
#endif

/* Planted mistakes, used only by the tests that show each pin catches one. */
enum {
    KDA_MUT_NONE = 0,
    KDA_MUT_DECAY_AFTER_WRITE = 1,   /* decay applied after the delta write   */
    KDA_MUT_OUTPUT_BEFORE_WRITE = 2, /* o_t read from the state before write  */
    KDA_MUT_DROP_BETA = 3,           /* write strength beta dropped           */
    KDA_MUT_SIGN = 4,                /* u = beta (v + S'^T k)                 */
    KDA_MUT_DECAY_ON_COLUMNS = 5     /* Diag(alpha) applied from the right    */
};

/* Returns 0 on success, 1 on bad arguments, 2 on allocation failure.
 * num_threads <= 0 uses every available core. */
int kda_oracle_fwd(int N, int H, int dk, int dv, const long long* cu_seqlens,
                   const double* q, const double* k, const double* v,
                   const double* log_alpha, const double* beta,
                   const double* initial_state, double scale, double* out,
                   double* final_state, int num_threads, int mutation);

int kda_oracle_max_threads(void);

#ifdef __cplusplus
}
#endif
#endif
