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
#include <math.h>
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

/*
 * Gradient of the recurrence (its exact vector-Jacobian product), for the
 * training backward pass that "Hardware-efficient implementation" (section 3
 * of paperlayer.ai/abs/2406.06484v6) runs after the forward: given the
 * upstream gradients dO of o and dS_T of S_T, it returns dq, dk, dv, dbeta
 * and dS_0 of L = <dO, o> + <dS_T, S_T>.
 *
 * Reverse mode through each token, with G = dL/dS_t (pages' orientation):
 *   o_t = S_t q_t                 G += dO_t q_t^T,   dq_t = S_t^T dO_t
 *   S_t = S_{t-1} + u_t k_t^T     du_t = G k_t,      dk_t (part) = G^T u_t
 *   u_t = beta_t e_t,             e_t = v_t - S_{t-1} k_t
 *                                 dv_t = beta_t du_t
 *                                 dbeta_t = <du_t, e_t>
 *                                 dk_t -= beta_t S_{t-1}^T du_t
 *                                 G  -= beta_t du_t k_t^T   (then G = dL/dS_{t-1})
 * Every state S_0 .. S_T of the head is kept (states[t] = S_t).
 */
static void grad_one_head(const double *q, const double *k, const double *v,
                          const double *beta, const double *S0, const double *dO,
                          const double *dST, double *dq, double *dk, double *dvv,
                          double *dbeta, double *dS0, long T, long dk_, long dv,
                          double *states, double *G, double *e, double *du)
{
    const size_t n = (size_t)dk_ * (size_t)dv;
    for (size_t x = 0; x < n; ++x)
        states[x] = S0 ? S0[x] : 0.0;
    for (long t = 0; t < T; ++t) {  /* forward, keeping S_t */
        const double *Sp = states + (size_t)t * n;
        double *St = states + (size_t)(t + 1) * n;
        const double *kt = k + t * dk_;
        for (long j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (long i = 0; i < dk_; ++i)
                acc += S_AT(Sp, dv, j, i) * kt[i];
            e[j] = v[t * dv + j] - acc;
        }
        for (long j = 0; j < dv; ++j)
            for (long i = 0; i < dk_; ++i)
                S_AT(St, dv, j, i) = S_AT(Sp, dv, j, i) + beta[t] * e[j] * kt[i];
    }
    for (size_t x = 0; x < n; ++x)
        G[x] = dST ? dST[x] : 0.0;
    for (long t = T - 1; t >= 0; --t) {
        const double *Sp = states + (size_t)t * n;
        const double *St = states + (size_t)(t + 1) * n;
        const double *kt = k + t * dk_, *qt = q + t * dk_, *dOt = dO + t * dv;
        const double bt = beta[t];
        /* read: o_t = S_t q_t */
        for (long j = 0; j < dv; ++j)
            for (long i = 0; i < dk_; ++i)
                S_AT(G, dv, j, i) += dOt[j] * qt[i];
        for (long i = 0; i < dk_; ++i) {
            double acc = 0.0;
            for (long j = 0; j < dv; ++j)
                acc += S_AT(St, dv, j, i) * dOt[j];
            dq[t * dk_ + i] = acc;
        }
        /* write: S_t = S_{t-1} + beta_t e_t k_t^T */
        for (long j = 0; j < dv; ++j) {
            double a = 0.0, p = 0.0;
            for (long i = 0; i < dk_; ++i) {
                a += S_AT(G, dv, j, i) * kt[i];
                p += S_AT(Sp, dv, j, i) * kt[i];
            }
            du[j] = a;
            e[j] = v[t * dv + j] - p;
        }
        double db = 0.0;
        for (long j = 0; j < dv; ++j) {
            dvv[t * dv + j] = bt * du[j];
            db += du[j] * e[j];
        }
        dbeta[t] = db;
        for (long i = 0; i < dk_; ++i) {
            double acc = 0.0;
            for (long j = 0; j < dv; ++j)
                acc += S_AT(G, dv, j, i) * bt * e[j] - bt * S_AT(Sp, dv, j, i) * du[j];
            dk[t * dk_ + i] = acc;
        }
        for (long j = 0; j < dv; ++j)
            for (long i = 0; i < dk_; ++i)
                S_AT(G, dv, j, i) -= bt * du[j] * kt[i];
    }
    for (size_t x = 0; x < n; ++x)
        dS0[x] = G[x];
}

/*
 * Gradients for all BH (batch, head) pairs, on nthreads OpenMP threads.
 * S0 and dST may be NULL (zeros).  Layouts as for dn_oracle_forward; dO is
 * [BH][T][dv], the outputs dq, dk [BH][T][dk], dv [BH][T][dv], dbeta
 * [BH][T], dS0 [BH][dk][dv].  Returns 0, or -1 if scratch memory could not
 * be had.
 */
int dn_oracle_backward(const double *q, const double *k, const double *v,
                       const double *beta, const double *S0, const double *dO,
                       const double *dST, double *dq, double *dk, double *dvv,
                       double *dbeta, double *dS0, long BH, long T, long dk_,
                       long dv, int nthreads)
{
    int failed = 0;
    const size_t n = (size_t)dk_ * (size_t)dv;
    if (nthreads < 1)
        nthreads = 1;
#pragma omp parallel num_threads(nthreads)
    {
        double *states = (double *)malloc(sizeof(double) * (n * (size_t)(T + 1) + n + 2 * (size_t)dv + 2));
        if (!states) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (long h = 0; h < BH; ++h) {
            if (!states)
                continue;
            double *G = states + n * (size_t)(T + 1);
            double *e = G + n, *du = e + dv + 1;
            grad_one_head(q + h * T * dk_, k + h * T * dk_, v + h * T * dv, beta + h * T,
                          S0 ? S0 + h * n : NULL, dO + h * T * dv, dST ? dST + h * n : NULL,
                          dq + h * T * dk_, dk + h * T * dk_, dvv + h * T * dv, dbeta + h * T,
                          dS0 + h * n, T, dk_, dv, states, G, e, du);
        }
        free(states);
    }
    return failed ? -1 : 0;
}

/*
 * Gated DeltaNet ("Gated DeltaNet", garden.houmin.site/infra/delta-net;
 * "Gated DeltaNet : oublier d'abord l'état entier", fr.news.hada.io/topic?id=31925):
 * a scalar keep rate alpha_t = exp(g_t) per token decays the whole state
 * before the delta rule, in the order the second page fixes:
 *   forget       S~ = alpha_t S_{t-1}
 *   predict      p = S~ k_t
 *   correct      u = beta_t (v_t - p)
 *   write        S_t = S~ + u k_t^T
 *   read         o_t = S_t q_t
 * i.e. S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T.
 * g is the log keep rate ([BH][T], fp64), as implementations store it.
 */
static void run_one_head_gated(const double *q, const double *k, const double *v,
                               const double *beta, const double *g, double *S, double *o,
                               long T, long dk, long dv, double *p)
{
    for (long t = 0; t < T; ++t) {
        const double *kt = k + t * dk;
        const double *qt = q + t * dk;
        const double *vt = v + t * dv;
        double *ot = o + t * dv;
        const double alpha = exp(g[t]);
        for (long j = 0; j < dv; ++j)           /* forget */
            for (long i = 0; i < dk; ++i)
                S_AT(S, dv, j, i) *= alpha;
        for (long j = 0; j < dv; ++j) {         /* predict */
            double acc = 0.0;
            for (long i = 0; i < dk; ++i)
                acc += S_AT(S, dv, j, i) * kt[i];
            p[j] = acc;
        }
        for (long j = 0; j < dv; ++j) {         /* correct and write */
            const double u = beta[t] * (vt[j] - p[j]);
            for (long i = 0; i < dk; ++i)
                S_AT(S, dv, j, i) += u * kt[i];
        }
        for (long j = 0; j < dv; ++j) {         /* read */
            double acc = 0.0;
            for (long i = 0; i < dk; ++i)
                acc += S_AT(S, dv, j, i) * qt[i];
            ot[j] = acc;
        }
    }
}

int dn_oracle_forward_gated(const double *q, const double *k, const double *v,
                            const double *beta, const double *g, double *S, double *o,
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
            run_one_head_gated(q + n * T * dk, k + n * T * dk, v + n * T * dv, beta + n * T,
                               g + n * T, S + n * dk * dv, o + n * T * dv, T, dk, dv, p);
        }
        free(p);
    }
    return failed ? -1 : 0;
}

/*
 * Gradient of the Gated DeltaNet recurrence above (its exact vector-Jacobian
 * product), the gated counterpart of grad_one_head: with the same upstream
 * gradients it also returns dg, the gradient of the log keep rates.  Reverse
 * mode through each token, in the reverse of the page's order, with
 * G = dL/dS_t and S~ = alpha_t S_{t-1}:
 *   read     o_t = S_t q_t            G += dO_t q_t^T,  dq_t = S_t^T dO_t
 *   write    S_t = S~ + u k_t^T       du = G k_t,       dk_t (part) = G^T u
 *   correct  u = beta_t e,            e = v_t - S~ k_t
 *                                     dv_t = beta_t du, dbeta_t = <du, e>
 *   predict                           dk_t -= beta_t S~^T du
 *                                     G -= beta_t du k_t^T   (now dL/dS~)
 *   forget   S~ = alpha_t S_{t-1}     dalpha = <G, S_{t-1}>, dg_t = alpha_t dalpha
 *                                     G *= alpha_t           (now dL/dS_{t-1})
 * Every state S_0 .. S_T of the head is kept (states[t] = S_t).
 */
static void grad_one_head_gated(const double *q, const double *k, const double *v,
                                const double *beta, const double *g, const double *S0,
                                const double *dO, const double *dST, double *dq, double *dk,
                                double *dvv, double *dbeta, double *dg, double *dS0, long T,
                                long dk_, long dv, double *states, double *G, double *e,
                                double *du)
{
    const size_t n = (size_t)dk_ * (size_t)dv;
    for (size_t x = 0; x < n; ++x)
        states[x] = S0 ? S0[x] : 0.0;
    for (long t = 0; t < T; ++t) {  /* forward, keeping S_t */
        const double *Sp = states + (size_t)t * n;
        double *St = states + (size_t)(t + 1) * n;
        const double *kt = k + t * dk_;
        const double alpha = exp(g[t]);
        for (long j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (long i = 0; i < dk_; ++i)
                acc += alpha * S_AT(Sp, dv, j, i) * kt[i];
            e[j] = v[t * dv + j] - acc;
        }
        for (long j = 0; j < dv; ++j)
            for (long i = 0; i < dk_; ++i)
                S_AT(St, dv, j, i) = alpha * S_AT(Sp, dv, j, i) + beta[t] * e[j] * kt[i];
    }
    for (size_t x = 0; x < n; ++x)
        G[x] = dST ? dST[x] : 0.0;
    for (long t = T - 1; t >= 0; --t) {
        const double *Sp = states + (size_t)t * n;
        const double *St = states + (size_t)(t + 1) * n;
        const double *kt = k + t * dk_, *qt = q + t * dk_, *dOt = dO + t * dv;
        const double bt = beta[t], alpha = exp(g[t]);
        /* read */
        for (long j = 0; j < dv; ++j)
            for (long i = 0; i < dk_; ++i)
                S_AT(G, dv, j, i) += dOt[j] * qt[i];
        for (long i = 0; i < dk_; ++i) {
            double acc = 0.0;
            for (long j = 0; j < dv; ++j)
                acc += S_AT(St, dv, j, i) * dOt[j];
            dq[t * dk_ + i] = acc;
        }
        /* write, correct, predict (S~ = alpha S_{t-1}) */
        for (long j = 0; j < dv; ++j) {
            double a = 0.0, p = 0.0;
            for (long i = 0; i < dk_; ++i) {
                a += S_AT(G, dv, j, i) * kt[i];
                p += alpha * S_AT(Sp, dv, j, i) * kt[i];
            }
            du[j] = a;
            e[j] = v[t * dv + j] - p;
        }
        double db = 0.0;
        for (long j = 0; j < dv; ++j) {
            dvv[t * dv + j] = bt * du[j];
            db += du[j] * e[j];
        }
        dbeta[t] = db;
        for (long i = 0; i < dk_; ++i) {
            double acc = 0.0;
            for (long j = 0; j < dv; ++j)
                acc += S_AT(G, dv, j, i) * bt * e[j] - bt * alpha * S_AT(Sp, dv, j, i) * du[j];
            dk[t * dk_ + i] = acc;
        }
        for (long j = 0; j < dv; ++j)
            for (long i = 0; i < dk_; ++i)
                S_AT(G, dv, j, i) -= bt * du[j] * kt[i];
        /* forget */
        double da = 0.0;
        for (size_t x = 0; x < n; ++x)
            da += G[x] * Sp[x];
        dg[t] = alpha * da;
        for (size_t x = 0; x < n; ++x)
            G[x] *= alpha;
    }
    for (size_t x = 0; x < n; ++x)
        dS0[x] = G[x];
}

/*
 * Gradients of the gated recurrence for all BH pairs (layouts as for
 * dn_oracle_backward; g and dg [BH][T]).  Returns 0, or -1 if scratch memory
 * could not be had.
 */
int dn_oracle_backward_gated(const double *q, const double *k, const double *v,
                             const double *beta, const double *g, const double *S0,
                             const double *dO, const double *dST, double *dq, double *dk,
                             double *dvv, double *dbeta, double *dg, double *dS0, long BH,
                             long T, long dk_, long dv, int nthreads)
{
    int failed = 0;
    const size_t n = (size_t)dk_ * (size_t)dv;
    if (nthreads < 1)
        nthreads = 1;
#pragma omp parallel num_threads(nthreads)
    {
        double *states = (double *)malloc(sizeof(double) * (n * (size_t)(T + 1) + n + 2 * (size_t)dv + 2));
        if (!states) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (long h = 0; h < BH; ++h) {
            if (!states)
                continue;
            double *G = states + n * (size_t)(T + 1);
            double *e = G + n, *du = e + dv + 1;
            grad_one_head_gated(q + h * T * dk_, k + h * T * dk_, v + h * T * dv, beta + h * T,
                                g + h * T, S0 ? S0 + h * n : NULL, dO + h * T * dv,
                                dST ? dST + h * n : NULL, dq + h * T * dk_, dk + h * T * dk_,
                                dvv + h * T * dv, dbeta + h * T, dg + h * T, dS0 + h * n, T,
                                dk_, dv, states, G, e, du);
        }
        free(states);
    }
    return failed ? -1 : 0;
}

/*
 * Kimi Delta Attention (KDA; "Kimi Delta Attention : atténuation par canal"
 * and "Transition diagonale-bas rang", fr.news.hada.io/topic?id=31925): the
 * scalar keep rate becomes one rate per key channel, alpha_t = exp(g_t) in
 * R^dk, D_t = Diag(alpha_t), in the order the page gives:
 *   decay        S~ = S_{t-1} D_t        (key channel i of S scaled by alpha_t[i])
 *   predict      p = S~ k_t
 *   correct      u = beta_t (v_t - p)
 *   write        S_t = S~ + u k_t^T
 *   read         o_t = S_t q_t          (the caller applies any query scale)
 * i.e. S_t = S_{t-1} D_t (I - beta_t k_t k_t^T) + beta_t v_t k_t^T.
 * g is [BH][T][dk] fp64 log keep rates.
 */
static void run_one_head_kda(const double *q, const double *k, const double *v,
                             const double *beta, const double *g, double *S, double *o,
                             long T, long dk, long dv, double *p)
{
    for (long t = 0; t < T; ++t) {
        const double *kt = k + t * dk, *qt = q + t * dk, *vt = v + t * dv, *gt = g + t * dk;
        double *ot = o + t * dv;
        for (long j = 0; j < dv; ++j)           /* decay, per key channel */
            for (long i = 0; i < dk; ++i)
                S_AT(S, dv, j, i) *= exp(gt[i]);
        for (long j = 0; j < dv; ++j) {         /* predict */
            double acc = 0.0;
            for (long i = 0; i < dk; ++i)
                acc += S_AT(S, dv, j, i) * kt[i];
            p[j] = acc;
        }
        for (long j = 0; j < dv; ++j) {         /* correct and write */
            const double u = beta[t] * (vt[j] - p[j]);
            for (long i = 0; i < dk; ++i)
                S_AT(S, dv, j, i) += u * kt[i];
        }
        for (long j = 0; j < dv; ++j) {         /* read */
            double acc = 0.0;
            for (long i = 0; i < dk; ++i)
                acc += S_AT(S, dv, j, i) * qt[i];
            ot[j] = acc;
        }
    }
}

int dn_oracle_forward_kda(const double *q, const double *k, const double *v,
                          const double *beta, const double *g, double *S, double *o,
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
            run_one_head_kda(q + n * T * dk, k + n * T * dk, v + n * T * dv, beta + n * T,
                             g + n * T * dk, S + n * dk * dv, o + n * T * dv, T, dk, dv, p);
        }
        free(p);
    }
    return failed ? -1 : 0;
}

/*
 * Gradient of the KDA recurrence above (its exact vector-Jacobian product),
 * the per-channel counterpart of grad_one_head_gated: the same reverse pass
 * through each token, in the reverse of the page's order, with G = dL/dS_t
 * and the decay S~ = S_{t-1} D_t scaling key channel i by alpha_t[i]:
 *   read     o_t = S_t q_t            G += dO_t q_t^T,  dq_t = S_t^T dO_t
 *   write    S_t = S~ + u k_t^T       du = G k_t,       dk_t (part) = G^T u
 *   correct  u = beta_t e,            e = v_t - S~ k_t
 *                                     dv_t = beta_t du, dbeta_t = <du, e>
 *   predict                           dk_t -= beta_t S~^T du
 *                                     G -= beta_t du k_t^T   (now dL/dS~)
 *   decay    S~ = S_{t-1} D_t         dalpha_t[i] = sum_j G[j][i] S_{t-1}[j][i],
 *                                     dg_t[i] = alpha_t[i] dalpha_t[i],
 *                                     G[j][i] *= alpha_t[i]  (now dL/dS_{t-1})
 * g and dg are [T][dk]; every state S_0 .. S_T of the head is kept.
 */
static void grad_one_head_kda(const double *q, const double *k, const double *v,
                              const double *beta, const double *g, const double *S0,
                              const double *dO, const double *dST, double *dq, double *dk,
                              double *dvv, double *dbeta, double *dg, double *dS0, long T,
                              long dk_, long dv, double *states, double *G, double *e,
                              double *du, double *alpha)
{
    const size_t n = (size_t)dk_ * (size_t)dv;
    for (size_t x = 0; x < n; ++x)
        states[x] = S0 ? S0[x] : 0.0;
    for (long t = 0; t < T; ++t) {  /* forward, keeping S_t */
        const double *Sp = states + (size_t)t * n;
        double *St = states + (size_t)(t + 1) * n;
        const double *kt = k + t * dk_;
        for (long i = 0; i < dk_; ++i)
            alpha[i] = exp(g[t * dk_ + i]);
        for (long j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (long i = 0; i < dk_; ++i)
                acc += alpha[i] * S_AT(Sp, dv, j, i) * kt[i];
            e[j] = v[t * dv + j] - acc;
        }
        for (long j = 0; j < dv; ++j)
            for (long i = 0; i < dk_; ++i)
                S_AT(St, dv, j, i) = alpha[i] * S_AT(Sp, dv, j, i) + beta[t] * e[j] * kt[i];
    }
    for (size_t x = 0; x < n; ++x)
        G[x] = dST ? dST[x] : 0.0;
    for (long t = T - 1; t >= 0; --t) {
        const double *Sp = states + (size_t)t * n;
        const double *St = states + (size_t)(t + 1) * n;
        const double *kt = k + t * dk_, *qt = q + t * dk_, *dOt = dO + t * dv;
        const double bt = beta[t];
        for (long i = 0; i < dk_; ++i)
            alpha[i] = exp(g[t * dk_ + i]);
        /* read */
        for (long j = 0; j < dv; ++j)
            for (long i = 0; i < dk_; ++i)
                S_AT(G, dv, j, i) += dOt[j] * qt[i];
        for (long i = 0; i < dk_; ++i) {
            double acc = 0.0;
            for (long j = 0; j < dv; ++j)
                acc += S_AT(St, dv, j, i) * dOt[j];
            dq[t * dk_ + i] = acc;
        }
        /* write, correct, predict (S~ = S_{t-1} D_t) */
        for (long j = 0; j < dv; ++j) {
            double a = 0.0, p = 0.0;
            for (long i = 0; i < dk_; ++i) {
                a += S_AT(G, dv, j, i) * kt[i];
                p += alpha[i] * S_AT(Sp, dv, j, i) * kt[i];
            }
            du[j] = a;
            e[j] = v[t * dv + j] - p;
        }
        double db = 0.0;
        for (long j = 0; j < dv; ++j) {
            dvv[t * dv + j] = bt * du[j];
            db += du[j] * e[j];
        }
        dbeta[t] = db;
        for (long i = 0; i < dk_; ++i) {
            double acc = 0.0;
            for (long j = 0; j < dv; ++j)
                acc += S_AT(G, dv, j, i) * bt * e[j] - bt * alpha[i] * S_AT(Sp, dv, j, i) * du[j];
            dk[t * dk_ + i] = acc;
        }
        for (long j = 0; j < dv; ++j)
            for (long i = 0; i < dk_; ++i)
                S_AT(G, dv, j, i) -= bt * du[j] * kt[i];
        /* decay, channel by channel */
        for (long i = 0; i < dk_; ++i) {
            double da = 0.0;
            for (long j = 0; j < dv; ++j)
                da += S_AT(G, dv, j, i) * S_AT(Sp, dv, j, i);
            dg[t * dk_ + i] = alpha[i] * da;
        }
        for (long j = 0; j < dv; ++j)
            for (long i = 0; i < dk_; ++i)
                S_AT(G, dv, j, i) *= alpha[i];
    }
    for (size_t x = 0; x < n; ++x)
        dS0[x] = G[x];
}

/*
 * Gradients of the KDA recurrence for all BH pairs (layouts as for
 * dn_oracle_backward; g and dg [BH][T][dk]).  Returns 0, or -1 if scratch
 * memory could not be had.
 */
int dn_oracle_backward_kda(const double *q, const double *k, const double *v,
                           const double *beta, const double *g, const double *S0,
                           const double *dO, const double *dST, double *dq, double *dk,
                           double *dvv, double *dbeta, double *dg, double *dS0, long BH,
                           long T, long dk_, long dv, int nthreads)
{
    int failed = 0;
    const size_t n = (size_t)dk_ * (size_t)dv;
    if (nthreads < 1)
        nthreads = 1;
#pragma omp parallel num_threads(nthreads)
    {
        double *states = (double *)malloc(sizeof(double) * (n * (size_t)(T + 1) + n +
                                                            2 * (size_t)dv + (size_t)dk_ + 2));
        if (!states) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (long h = 0; h < BH; ++h) {
            if (!states)
                continue;
            double *G = states + n * (size_t)(T + 1);
            double *e = G + n, *du = e + dv + 1, *alpha = du + dv + 1;
            grad_one_head_kda(q + h * T * dk_, k + h * T * dk_, v + h * T * dv, beta + h * T,
                              g + h * T * dk_, S0 ? S0 + h * n : NULL, dO + h * T * dv,
                              dST ? dST + h * n : NULL, dq + h * T * dk_, dk + h * T * dk_,
                              dvv + h * T * dv, dbeta + h * T, dg + h * T * dk_, dS0 + h * n, T,
                              dk_, dv, states, G, e, du, alpha);
        }
        free(states);
    }
    return failed ? -1 : 0;
}

/*
 * Optional input preparation ahead of any of the forms above, one row of
 * length d at a time:
 *
 *   normalised   y = x / sqrt(sum_i x_i^2 + eps)     (when normalize != 0)
 *   scaled       y = scale * y
 *
 * The normalisation is the l2norm helper of the Gated DeltaNet PyTorch code
 * on "DeltaNet 引入 Delta Rule" (garden.houmin.site/infra/delta-net), which
 * normalises queries and keys over the head dimension with eps = 1e-6 and
 * divides the queries by the square root of the head dimension; the layer of
 * "fla/layers/delta_net.py" asks its kernels for the same normalisation
 * (use_qk_l2norm_in_kernel).  The KDA read of "Kimi Delta Attention"
 * (fr.news.hada.io/topic?id=31925) scales q by d_k^{-1/2}.  The queries get
 * the scale, the keys do not.
 *   x, y   [rows][d]   (y may equal x)
 */
void dn_oracle_prepare_rows(const double *x, double *y, long rows, long d,
                            int normalize, double scale, double eps)
{
    for (long r = 0; r < rows; ++r) {
        const double *xr = x + r * d;
        double *yr = y + r * d;
        double f = scale;
        if (normalize) {
            double ss = 0.0;
            for (long i = 0; i < d; ++i)
                ss += xr[i] * xr[i];
            f = scale / sqrt(ss + eps);
        }
        for (long i = 0; i < d; ++i)
            yr[i] = xr[i] * f;
    }
}

/*
 * Gradient of the preparation above, per row: given the row x and the
 * gradient dy of its output y = scale * x / n (n = sqrt(sum x^2 + eps)),
 *
 *   dx = (scale / n) (dy - x (x . dy) / n^2)     (normalize != 0)
 *   dx = scale dy                                (normalize == 0)
 *
 * which is the chain rule through y_i = scale x_i / n with
 * dn/dx_i = x_i / n.  x, dy, dx are [rows][d] (dx may equal dy).
 */
void dn_oracle_prepare_rows_backward(const double *x, const double *dy, double *dx,
                                     long rows, long d, int normalize, double scale,
                                     double eps)
{
    for (long r = 0; r < rows; ++r) {
        const double *xr = x + r * d;
        const double *gr = dy + r * d;
        double *out = dx + r * d;
        if (!normalize) {
            for (long i = 0; i < d; ++i)
                out[i] = scale * gr[i];
            continue;
        }
        double ss = 0.0, xg = 0.0;
        for (long i = 0; i < d; ++i) {
            ss += xr[i] * xr[i];
            xg += xr[i] * gr[i];
        }
        const double n2 = ss + eps;
        const double n = sqrt(n2);
        for (long i = 0; i < d; ++i)
            out[i] = scale / n * (gr[i] - xr[i] * xg / n2);
    }
}
