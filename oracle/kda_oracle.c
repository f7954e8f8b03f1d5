/*
 * kda_oracle.c -- fp64 CPU oracle of the Kimi Delta Attention (KDA) layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark do.  It shares no code, header or constant table with the
 * CUDA library.
 *
 * What it computes (plain definitions, no blocking, no reordering):
 *
 *   gate   g_t = g_min * sigmoid(exp(A) (.) z_t),  g_min = -5,  alpha_t = exp(g_t)
 *          -- "How Kimi K3 is built: 2.8 trillion parameters, linear attention
 *             and agents for a million tokens", section "Sequence: three KDA to
 *             one global MLA"; the bound alpha in [e^-5, 1] is restated in
 *             "Kimi K3 architecture: how an open model with a million-token
 *             context competes with market leaders", section "How the Kimi K3
 *             architecture holds a million tokens of context".
 *
 *   state  S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *   output o_t = S_t^T q_t
 *          -- the delta rule of the second page above, same section (a fixed
 *             state S that each token partially erases and then writes; beta =
 *             write strength, alpha = forget factor applied before the write),
 *             with the per-channel forget gate of the first page above (the
 *             channel-wise coefficient decides what is kept before the write).
 *             Decay first, then erase, then write; o_t reads the state after
 *             the update.
 *
 * Per (sequence, head) the recurrence is evaluated token by token in fp64.
 * Inputs are read in their stored type (fp32 or bf16) and converted exactly to
 * double one token at a time, so no fp64 copy of a whole tensor is made.
 * Independent (sequence, head) pairs are spread over POSIX threads.
 *
 * Layouts (row-major): q, k, z [T_total, H, dk]; v [T_total, H, dv];
 * beta [T_total, H]; A [H, dk] fp32; S0 [N, H, dk, dv] fp32 (nullable).
 * A fixed-length batch [B, T, ...] is the packed case with
 * cu_seqlens = {0, T, 2T, ..., B*T}.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define KDA_REF_GMIN (-5.0)

enum { REF_F32 = 0, REF_BF16 = 1 };

static double ref_load(const void *p, int64_t i, int dtype)
{
    if (dtype == REF_BF16) {
        uint16_t h = ((const uint16_t *)p)[i];
        uint32_t u = (uint32_t)h << 16;
        float f;
        memcpy(&f, &u, sizeof f);
        return (double)f;
    }
    return (double)((const float *)p)[i];
}

/* g = g_min * sigmoid(exp(A) * z), sigmoid(x) = 1 / (1 + exp(-x)). */
double kda_ref_gate_scalar(double a, double z)
{
    double x = exp(a) * z;
    double sig = 1.0 / (1.0 + exp(-x));
    return KDA_REF_GMIN * sig;
}

/* g_out[t, h, c] = gate(A[h, c], z[t, h, c]) for every token. */
void kda_ref_gate(const void *z, int dtype, const float *A, double *g_out,
                  int64_t n_tokens, int H, int dk)
{
    for (int64_t t = 0; t < n_tokens; ++t)
        for (int h = 0; h < H; ++h)
            for (int c = 0; c < dk; ++c) {
                int64_t i = (t * H + h) * dk + c;
                g_out[i] = kda_ref_gate_scalar((double)A[h * dk + c], ref_load(z, i, dtype));
            }
}

typedef struct {
    const void *q, *k, *v, *z, *beta;
    int dtype;
    const float *A;
    const float *S0;
    const int64_t *cu;
    int H, dk, dv;
    const int64_t *pairs;   /* [n_pairs, 2] = (seq, head) */
    int64_t n_pairs;
    const int64_t *o_off;   /* start of each pair's block in o_out */
    double *o_out;          /* per pair [len, dv]; may be NULL */
    double *S_out;          /* per pair [dk, dv]; may be NULL */
    int64_t next;           /* shared work counter */
} ref_job;

/* One (sequence, head): the recurrence exactly as written above. */
static void ref_run_pair(const ref_job *J, int64_t p, double *S, double *D,
                         double *kv, double *qv, double *alpha, double *vv, double *kD)
{
    const int64_t n = J->pairs[2 * p], h = J->pairs[2 * p + 1];
    const int H = J->H, dk = J->dk, dv = J->dv;
    const int64_t bos = J->cu[n], eos = J->cu[n + 1];

    for (int c = 0; c < dk; ++c)
        for (int j = 0; j < dv; ++j)
            S[c * dv + j] = J->S0 ? (double)J->S0[((n * H + h) * dk + c) * dv + j] : 0.0;

    double *o = J->o_out ? J->o_out + J->o_off[p] : NULL;
    for (int64_t t = bos; t < eos; ++t) {
        const int64_t row = t * H + h;
        for (int c = 0; c < dk; ++c) {
            kv[c] = ref_load(J->k, row * dk + c, J->dtype);
            qv[c] = ref_load(J->q, row * dk + c, J->dtype);
            alpha[c] = exp(kda_ref_gate_scalar((double)J->A[h * dk + c],
                                               ref_load(J->z, row * dk + c, J->dtype)));
        }
        for (int j = 0; j < dv; ++j)
            vv[j] = ref_load(J->v, row * dv + j, J->dtype);
        const double b = ref_load(J->beta, row, J->dtype);

        /* D = Diag(alpha_t) S_{t-1} */
        for (int c = 0; c < dk; ++c)
            for (int j = 0; j < dv; ++j)
                D[c * dv + j] = alpha[c] * S[c * dv + j];
        /* kD = k_t^T D  (a row vector over dv) */
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int c = 0; c < dk; ++c)
                acc += kv[c] * D[c * dv + j];
            kD[j] = acc;
        }
        /* S_t = D - beta k (k^T D) + beta k v^T = (I - beta k k^T) D + beta k v^T */
        for (int c = 0; c < dk; ++c)
            for (int j = 0; j < dv; ++j)
                S[c * dv + j] = D[c * dv + j] - b * kv[c] * kD[j] + b * kv[c] * vv[j];
        /* o_t = S_t^T q_t */
        if (o) {
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int c = 0; c < dk; ++c)
                    acc += S[c * dv + j] * qv[c];
                o[(t - bos) * dv + j] = acc;
            }
        }
    }
    if (J->S_out)
        memcpy(J->S_out + p * (int64_t)dk * dv, S, sizeof(double) * (size_t)dk * dv);
}

static void *ref_worker(void *arg)
{
    ref_job *J = (ref_job *)arg;
    const size_t sd = (size_t)J->dk * J->dv;
    double *buf = (double *)malloc(sizeof(double) * (2 * sd + 3 * (size_t)J->dk + 2 * (size_t)J->dv));
    if (!buf)
        return (void *)1;
    double *S = buf, *D = S + sd, *kv = D + sd, *qv = kv + J->dk, *alpha = qv + J->dk;
    double *vv = alpha + J->dk, *kD = vv + J->dv;
    for (;;) {
        int64_t p = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
        if (p >= J->n_pairs)
            break;
        ref_run_pair(J, p, S, D, kv, qv, alpha, vv, kD);
    }
    free(buf);
    return NULL;
}

/*
 * Runs the recurrence for the listed (sequence, head) pairs.
 *   pairs   [n_pairs, 2] int64 (seq index into cu_seqlens, head index)
 *   o_out   nullable; pair p's outputs [len_p, dv] start at the sum of the
 *           earlier pairs' len * dv (pairs laid out back to back, in order)
 *   S_out   nullable; [n_pairs, dk, dv] final states
 *   n_threads <= 0 means one thread per online core.
 * Returns 0 on success, -1 on bad arguments or allocation failure.
 */
int kda_ref_recurrent(const void *q, const void *k, const void *v, const void *z,
                      const void *beta, int dtype, const float *A, const float *S0,
                      const int64_t *cu_seqlens, int64_t n_seqs, int H, int dk, int dv,
                      const int64_t *pairs, int64_t n_pairs, double *o_out, double *S_out,
                      int n_threads)
{
    if (!q || !k || !v || !z || !beta || !A || !cu_seqlens || !pairs || H <= 0 || dk <= 0 ||
        dv <= 0 || n_pairs < 0 || (dtype != REF_F32 && dtype != REF_BF16))
        return -1;
    for (int64_t p = 0; p < n_pairs; ++p)
        if (pairs[2 * p] < 0 || pairs[2 * p] >= n_seqs || pairs[2 * p + 1] < 0 ||
            pairs[2 * p + 1] >= H)
            return -1;

    int64_t *off = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n_pairs + 1));
    if (!off)
        return -1;
    off[0] = 0;
    for (int64_t p = 0; p < n_pairs; ++p) {
        int64_t n = pairs[2 * p];
        off[p + 1] = off[p] + (cu_seqlens[n + 1] - cu_seqlens[n]) * dv;
    }

    ref_job J = {q, k, v, z, beta, dtype, A, S0, cu_seqlens, H, dk, dv,
                 pairs, n_pairs, off, o_out, S_out, 0};
    if (n_threads <= 0)
        n_threads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (n_threads < 1)
        n_threads = 1;
    if (n_threads > n_pairs)
        n_threads = n_pairs > 0 ? (int)n_pairs : 1;

    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    int rc = 0;
    if (!th) {
        free(off);
        return -1;
    }
    int started = 0;
    for (int i = 0; i < n_threads; ++i) {
        if (pthread_create(&th[i], NULL, ref_worker, &J) != 0)
            break;
        ++started;
    }
    if (started == 0)
        rc = (ref_worker(&J) == NULL) ? 0 : -1;
    for (int i = 0; i < started; ++i) {
        void *ret = NULL;
        pthread_join(th[i], &ret);
        if (ret)
            rc = -1;
    }
    free(th);
    free(off);
    return rc;
}

/* Number of online cores the oracle's default thread count uses. */
int kda_ref_default_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}
