/*
 * deltanet_oracle.c -- TEST INFRASTRUCTURE, NOT PRODUCT CODE.
 *
 * A plain, slow, fp64 CPU statement of the DeltaNet delta-rule recurrence,
 * used only to check the CUDA path.  Only tests, the smoke check and the
 * benchmark's CPU-baseline leg may load it.  It shares no code, header or
 * constant with the CUDA library.
 *
 * What it computes (per batch b and head h, independently, token by token):
 *
 *   prediction   p_t = S_{t-1} k_t
 *   error        u_t = beta_t (v_t - p_t)
 *   write        S_t = S_{t-1} + u_t k_t^T
 *   read         o_t = S_t q_t            (the read comes after the write)
 *
 * Sources:
 *   - "DeltaNet 引入 Delta Rule" (garden.houmin.site/infra/delta-net): the
 *     error-correcting form S_t = S_{t-1} - beta_t (S_{t-1} k_t - v_t) k_t^T and
 *     the read o_t = S_t q_t.
 *   - "DeltaNet : écrire l'erreur de prédiction plutôt que la valeur"
 *     (fr.news.hada.io/topic?id=31925): e_t = beta_t (v_t - S_{t-1} k_t),
 *     S_t = S_{t-1} + e_t k_t^T.
 *   - "Calcul de toutes les sorties internes au chunk" on the same page: a
 *     token's output includes its own write.
 *
 * Notation: the pages' state S maps key space to value space, so S is
 * dv x dk and S(j,i) multiplies key channel i into value channel j.  In
 * memory the state is stored transposed, as [dk][dv] (value channel
 * contiguous), which is the layout the library's callers use; the accessor
 * below hides that so the loops read like the pages.
 *
 * Layouts (all contiguous fp64):
 *   q, k   [BH][T][dk]      v, o  [BH][T][dv]      beta  [BH][T]
 *   S      [BH][dk][dv]     holds S_0 on entry and S_T on return.
 * BH is the number of independent (batch, head) pairs.
 */
#include <stdlib.h>

/* The pages' S(j,i) for a state stored as [dk][dv]. */
#define S_AT(S, dv, j, i) ((S)[(size_t)(i) * (size_t)(dv) + (size_t)(j)])

/* Runs the recurrence over T tokens for one (batch, head). */
static void run_one_head(const double *q, const double *k, const double *v,
                         const double *beta, double *S, double *o,
                         long T, long dk, long dv, double *p)
{
    for (long t = 0; t < T; ++t) {
        const double *kt = k + t * dk;
        const double *qt = q + t * dk;
        const double *vt = v + t * dv;
        double *ot = o + t * dv;
        const double bt = beta[t];

        /* prediction p = S_{t-1} k_t */
        for (long j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (long i = 0; i < dk; ++i)
                acc += S_AT(S, dv, j, i) * kt[i];
            p[j] = acc;
        }
        /* error u = beta_t (v_t - p), written as S += u k_t^T */
        for (long j = 0; j < dv; ++j) {
            const double u = bt * (vt[j] - p[j]);
            for (long i = 0; i < dk; ++i)
                S_AT(S, dv, j, i) += u * kt[i];
        }
        /* read o_t = S_t q_t */
        for (long j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (long i = 0; i < dk; ++i)
                acc += S_AT(S, dv, j, i) * qt[i];
            ot[j] = acc;
        }
    }
}

/*
 * Runs all BH (batch, head) pairs on nthreads OpenMP threads (values below 1
 * mean one thread).  Returns 0, or -1 if scratch memory could not be had.
 */
int dn_oracle_forward(const double *q, const double *k, const double *v,
                      const double *beta, double *S, double *o,
                      long BH, long T, long dk, long dv, int nthreads)
{
    int failed = 0;
    if (nthreads < 1)
        nthreads = 1;
#pragma omp parallel num_threads(nthreads)
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)(dv > 0 ? dv : 1));
        if (!p) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (long n = 0; n < BH; ++n) {
            if (!p)
                continue;
            run_one_head(q + n * T * dk, k + n * T * dk, v + n * T * dv,
                         beta + n * T, S + n * dk * dv, o + n * T * dv,
                         T, dk, dv, p);
        }
        free(p);
    }
    return failed ? -1 : 0;
}
