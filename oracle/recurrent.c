/*
 * Simple GLA oracle: the step-by-step recurrence, in fp64, on host threads.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the reference that the GPU path is checked
 * against. Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load it. It shares no code, header or constant with the CUDA library.
 *
 * What it computes, per sequence n and head h, starting from S = h0[n,h] (or zeros):
 *
 *   for each token t of sequence n, in order:
 *     alpha = exp(g[t,h])                      (decay, step 1)
 *     S     = alpha * S                        (step 1)
 *     S     = S + k[t,h]^T (outer) v[t,h]      (update, step 2; k indexes the rows of S)
 *     o[t,h][j] = scale * sum_i q[t,h][i] * S[i][j]   (query, step 3)
 *   hT[n,h] = S
 *
 * Source: "MiniCPM-SALA — Complete Blueprint", section "B2 lightning-attn (Simple GLA)",
 * block "Simple GLA Recurrence" (steps 1 decay, 2 outer-product update, 3 query times the
 * 1/sqrt(128) scale, in that order; the state is [d_k x d_v] because k^T is [128,1] and v
 * is [1,128]). The per-token log-decay g[t,h] generalises the page's per-head constant
 * g_gamma[h]; "Formulas and Code for Adapting Inference to GDN/KDA Linear Modules",
 * section 1.1 (recursive form), has the same loop with a per-token gate, of which this is
 * the special case without the delta term and with beta = 1.
 *
 * Inputs are the exact values the GPU receives: q, k, v as raw bfloat16 bit patterns,
 * g as float32, h0 as float64 (widened by the caller from float32). Every product and
 * sum is done in double precision; outputs stay double.
 *
 * Layouts (row-major, last index contiguous):
 *   q, k : [T_total, H, dk]   bf16 bits     v : [T_total, H, dv]  bf16 bits
 *   g    : [T_total, H]       float32
 *   cu_seqlens : [nseq + 1]   int64, sequence n owns tokens [cu[n], cu[n+1])
 *   heads      : [nh] int64 head indices to evaluate (NULL: all H heads, nh = H)
 *   h0   : [nseq, H, dk, dv]  float64 or NULL (zeros)
 *   o    : [T_total, nh, dv]  float64 or NULL (not written)
 *   hT   : [nseq, nh, dk, dv] float64 or NULL (not written)
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double widen_bf16(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16; /* bf16 is the top half of an IEEE float32 */
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

typedef struct {
    const uint16_t *q, *k, *v;
    const float *g;
    double scale;
    const double *h0;
    const int64_t *cu_seqlens;
    const int64_t *heads;
    int64_t nseq, H, nh, dk, dv;
    double *o, *hT;
    int64_t next_unit; /* shared work counter, guarded by lock */
    pthread_mutex_t lock;
} job_t;

static void run_unit(const job_t *a, int64_t n, int64_t hs, double *S, double *qd, double *kd,
                     double *vd)
{
    const int64_t H = a->H, dk = a->dk, dv = a->dv;
    const int64_t h = a->heads ? a->heads[hs] : hs;
    const int64_t bos = a->cu_seqlens[n], eos = a->cu_seqlens[n + 1];

    if (a->h0)
        memcpy(S, a->h0 + ((n * H + h) * dk) * dv, (size_t)(dk * dv) * sizeof(double));
    else
        memset(S, 0, (size_t)(dk * dv) * sizeof(double));

    for (int64_t t = bos; t < eos; ++t) {
        const int64_t row = t * H + h;
        for (int64_t i = 0; i < dk; ++i) {
            qd[i] = widen_bf16(a->q[row * dk + i]);
            kd[i] = widen_bf16(a->k[row * dk + i]);
        }
        for (int64_t j = 0; j < dv; ++j)
            vd[j] = widen_bf16(a->v[row * dv + j]);

        /* step 1: decay the whole state by alpha = exp(g) */
        const double alpha = exp((double)a->g[row]);
        for (int64_t i = 0; i < dk * dv; ++i)
            S[i] *= alpha;

        /* step 2: add the outer product k^T v (row i of S gets k_i * v) */
        for (int64_t i = 0; i < dk; ++i)
            for (int64_t j = 0; j < dv; ++j)
                S[i * dv + j] += kd[i] * vd[j];

        /* step 3: o_j = scale * sum_i q_i S[i][j], read after this token's update */
        if (a->o) {
            double *orow = a->o + (t * a->nh + hs) * dv;
            for (int64_t j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int64_t i = 0; i < dk; ++i)
                    acc += qd[i] * S[i * dv + j];
                orow[j] = a->scale * acc;
            }
        }
    }
    if (a->hT)
        memcpy(a->hT + ((n * a->nh + hs) * dk) * dv, S, (size_t)(dk * dv) * sizeof(double));
}

static void *worker(void *p)
{
    job_t *a = (job_t *)p;
    const int64_t units = a->nseq * a->nh;
    double *S = (double *)malloc((size_t)(a->dk * a->dv) * sizeof(double));
    double *qd = (double *)malloc((size_t)a->dk * sizeof(double));
    double *kd = (double *)malloc((size_t)a->dk * sizeof(double));
    double *vd = (double *)malloc((size_t)a->dv * sizeof(double));
    if (S && qd && kd && vd) {
        for (;;) {
            pthread_mutex_lock(&a->lock);
            const int64_t u = a->next_unit++;
            pthread_mutex_unlock(&a->lock);
            if (u >= units)
                break;
            run_unit(a, u / a->nh, u % a->nh, S, qd, kd, vd);
        }
    }
    free(S);
    free(qd);
    free(kd);
    free(vd);
    return NULL;
}

/* Returns 0 on success, a negative value on a bad argument or allocation failure. */
int oracle_recurrent(const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *g,
                     double scale, const double *h0, const int64_t *cu_seqlens, int64_t nseq,
                     int64_t H, int64_t dk, int64_t dv, const int64_t *heads, int64_t nh,
                     double *o, double *hT, int nthreads)
{
    if (!cu_seqlens || nseq < 0 || H < 1 || dk < 1 || dv < 1)
        return -1;
    if (!heads)
        nh = H;
    if (nh < 1)
        return -1;
    for (int64_t n = 0; n < nseq; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n])
            return -2;
    if (heads)
        for (int64_t i = 0; i < nh; ++i)
            if (heads[i] < 0 || heads[i] >= H)
                return -3;
    const int64_t T = nseq > 0 ? cu_seqlens[nseq] : 0;
    if (T > 0 && (!q || !k || !v || !g))
        return -1;

    job_t job = {q, k, v, g, scale, h0, cu_seqlens, heads, nseq, H, nh, dk, dv, o, hT, 0};
    pthread_mutex_init(&job.lock, NULL);
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    pthread_t tid[256];
    int started = 0;
    for (int i = 1; i < nthreads; ++i)
        if (pthread_create(&tid[started], NULL, worker, &job) == 0)
            ++started;
    worker(&job);
    for (int i = 0; i < started; ++i)
        pthread_join(tid[i], NULL);
    pthread_mutex_destroy(&job.lock);
    return 0;
}
