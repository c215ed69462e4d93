/*
 * Float64 CPU oracle for the Gated DeltaNet prefill -- TEST INFRASTRUCTURE.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this.  The product (the CUDA library) never calls it and shares no
 * code with it.
 *
 * What it computes.  The pages name a "chunked Gated DeltaNet prefill" that is
 * checked against float64 references ("Cua-S1 4B 0.2 native text worker",
 * kernel-test paragraph; "Open-Jev-27B-v1.1 native text worker", section
 * "Validation and optimization scope"), but print no equations.  This file
 * writes out the plain definition of the gated delta rule, token by token,
 * per (sequence, value head), with no chunking:
 *
 *     S_t = alpha_t * S_{t-1} * (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *     o_t = S_t q_t / sqrt(dk)
 *
 * with alpha_t = exp(g_t), S a dv x dk matrix (row i holds the weights that
 * produce output coordinate i), S_0 = init_state (zeros if NULL) and the last
 * S returned as the final state.  The update is evaluated in the algebraically
 * identical rank-one form
 *
 *     S <- alpha_t S;   u = beta_t (v_t - S k_t);   S <- S + u k_t^T
 *
 * (expanding alpha S (I - beta k k^T) + beta v k^T gives exactly this).
 *
 * Layouts (token-major, contiguous): q, k [Ttot, Hk, dk]; v, out [Ttot, Hv, dv];
 * g, beta [Ttot, Hv]; init_state, final_state [B, Hv, dv, dk].  Value head h
 * reads key head h / (Hv / Hk).  With cu_seqlens == NULL there are B sequences
 * of T tokens; otherwise sequence b covers tokens [cu_seqlens[b], cu_seqlens[b+1]).
 *
 * Work is spread over threads by (sequence, value head) pair; each pair is an
 * independent recurrence, so the result does not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    const double *q, *k, *v, *g, *beta, *init;
    const int32_t *cu;
    double *out, *fin;
    int B, T, Hk, Hv, dk, dv;
    int next; /* next (sequence, head) pair to take */
} job_t;

static void one_pair(const job_t *J, int n, int h, double *S)
{
    const int dk = J->dk, dv = J->dv, Hk = J->Hk, Hv = J->Hv;
    const int hk = h / (Hv / Hk);
    const double scale = 1.0 / sqrt((double)dk);
    long bos, eos;
    if (J->cu) {
        bos = J->cu[n];
        eos = J->cu[n + 1];
    } else {
        bos = (long)n * J->T;
        eos = bos + J->T;
    }
    if (J->init)
        memcpy(S, J->init + ((long)n * Hv + h) * dv * dk, sizeof(double) * dv * dk);
    else
        memset(S, 0, sizeof(double) * dv * dk);

    for (long t = bos; t < eos; ++t) {
        const double *kt = J->k + (t * Hk + hk) * dk;
        const double *qt = J->q + (t * Hk + hk) * dk;
        const double *vt = J->v + (t * Hv + h) * dv;
        const double alpha = exp(J->g[t * Hv + h]);
        const double beta = J->beta[t * Hv + h];
        double *ot = J->out + (t * Hv + h) * dv;
        for (int i = 0; i < dv; ++i) {
            double *Si = S + (long)i * dk;
            double sk = 0.0;
            for (int j = 0; j < dk; ++j) {
                Si[j] *= alpha;          /* decay */
                sk += Si[j] * kt[j];     /* (alpha S) k */
            }
            const double u = beta * (vt[i] - sk);
            double sq = 0.0;
            for (int j = 0; j < dk; ++j) {
                Si[j] += u * kt[j];      /* rank-one write */
                sq += Si[j] * qt[j];     /* S_t q_t */
            }
            ot[i] = sq * scale;
        }
    }
    if (J->fin)
        memcpy(J->fin + ((long)n * Hv + h) * dv * dk, S, sizeof(double) * dv * dk);
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    double *S = (double *)malloc(sizeof(double) * J->dv * J->dk);
    if (!S)
        return (void *)1;
    const int npairs = J->B * J->Hv;
    for (;;) {
        int p = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
        if (p >= npairs)
            break;
        one_pair(J, p / J->Hv, p % J->Hv, S);
    }
    free(S);
    return NULL;
}

int gdn_oracle_num_cpus(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/* Returns 0 on success, -1 on bad arguments, -2 when threads or memory fail.
 * nthreads <= 0 means one thread per online CPU. */
int gdn_oracle_prefill(const double *q, const double *k, const double *v,
                       const double *g, const double *beta,
                       const int32_t *cu_seqlens, const double *init_state,
                       double *out, double *final_state,
                       int B, int T, int Hk, int Hv, int dk, int dv, int nthreads)
{
    if (B < 0 || T < 0 || Hk <= 0 || Hv <= 0 || Hv % Hk || dk <= 0 || dv <= 0)
        return -1;
    if (!q || !k || !v || !g || !beta || !out)
        return -1;
    job_t J = {q, k, v, g, beta, init_state, cu_seqlens, out, final_state,
               B, T, Hk, Hv, dk, dv, 0};
    int npairs = B * Hv;
    if (npairs == 0)
        return 0;
    if (nthreads <= 0)
        nthreads = gdn_oracle_num_cpus();
    if (nthreads > npairs)
        nthreads = npairs;
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!th)
        return -2;
    int rc = 0, started = 0;
    for (int i = 0; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, worker, &J) != 0) {
            rc = -2;
            break;
        }
        ++started;
    }
    for (int i = 0; i < started; ++i) {
        void *ret = NULL;
        pthread_join(th[i], &ret);
        if (ret)
            rc = -2;
    }
    free(th);
    if (started == 0)
        rc = -2;
    return rc;
}
