/*
 * Float64 CPU oracle for the fused grouped-query attention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only tests/, the smoke check in __graft_entry__.py and the
 * cpu_baseline / reference legs of bench.py use it.  It shares no code,
 * header, table or helper with the CUDA kernels.
 *
 * What it computes is the plain definition of attention as written on the
 * page "从零开始写Qwen3" (deepseek.csdn.net/6a3201f8..., the derivation page),
 * section "简易情况-三矩阵相乘", the softmax form of O:
 *
 *     s_ij  = scale * <q_i, k_j>                        (scores, materialised)
 *     s_ij  = -inf  where the causal mask forbids j > i  (section "FlashAttention",
 *                                                         mask(Q_i K_j^T / sqrt(D)))
 *     m_i   = max_j s_ij
 *     p_ij  = exp(s_ij - m_i),   l_i = sum_j p_ij
 *     o_i   = sum_j p_ij v_j / l_i
 *     lse_i = m_i + ln(l_i)                              (natural log)
 *
 * Grouped-query heads follow the same page's kernel, section "FlashAttention":
 * the flattened (b, q_head) index divided by the group size gives the
 * flattened (b, kv_head) index, i.e. kv_head = q_head / (Hq / Hkv) with the
 * batch kept.  There is no tiling, no online rescaling and no fusion here:
 * one full score row per (b, q_head, i) in float64.
 *
 * Queries and keys may differ in number: Nq query rows attend over Nk keys
 * (that page's kernel keeps separate query and key lengths).  The causal mask
 * is then aligned at the bottom right: query i sees key j when
 * j <= i + (Nk - Nq), so the query rows are the last Nq positions of an
 * Nk-token sequence.  With Nq == Nk this is the square mask j <= i.  A causal
 * call needs Nq <= Nk, so that every query row sees at least key 0.
 *
 * Layouts (row-major, float64): q, o [B, Hq, Nq, D]; k, v [B, Hkv, Nk, D];
 * lse [B, Hq, Nq].
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <unistd.h>

/* One output row: (b, hq, i).  qi points at the D query values of the row;
 * kh, vh at the [N, D] key / value matrices of the row's kv head (N = Nk);
 * off = Nk - Nq is the causal alignment offset.  s is an N-long scratch row. */
static void attend_row(const double *qi, const double *kh, const double *vh,
                       long i, long N, long D, double scale, int causal,
                       long off, double *s, double *oi, double *lse_i)
{
    long j, d;
    /* scores with the mask applied as -inf */
    for (j = 0; j < N; ++j) {
        double acc = 0.0;
        if (causal && j > i + off) {
            s[j] = -INFINITY;
            continue;
        }
        for (d = 0; d < D; ++d)
            acc += qi[d] * kh[j * D + d];
        s[j] = scale * acc;
    }
    /* softmax over the full row */
    double m = -INFINITY;
    for (j = 0; j < N; ++j)
        if (s[j] > m)
            m = s[j];
    double l = 0.0;
    for (j = 0; j < N; ++j) {
        double p = exp(s[j] - m);
        s[j] = p;
        l += p;
    }
    /* weighted sum of value rows, normalised once */
    for (d = 0; d < D; ++d)
        oi[d] = 0.0;
    for (j = 0; j < N; ++j) {
        if (s[j] == 0.0)
            continue; /* masked: weight exactly zero */
        for (d = 0; d < D; ++d)
            oi[d] += s[j] * vh[j * D + d];
    }
    for (d = 0; d < D; ++d)
        oi[d] = oi[d] / l;
    *lse_i = m + log(l);
}

typedef struct {
    const double *q_rows; /* [n_rows, D] query rows, in the order of rows[] */
    const long long *rows; /* flattened (b*Hq + hq)*Nq + i for each row */
    long n_rows;
    const double *k, *v;
    double *o_rows, *lse_rows;
    long Hq, Hkv, Nq, Nk, D;
    double scale;
    int causal;
    int tid, nthreads;
    int failed;
} job_t;

static void *run_rows(void *arg)
{
    job_t *J = (job_t *)arg;
    long group = J->Hq / J->Hkv;
    double *s = (double *)malloc(sizeof(double) * (size_t)J->Nk);
    if (!s) {
        J->failed = 1;
        return NULL;
    }
    /* interleaved split: causal rows have uneven cost, neighbours even it out */
    for (long r = J->tid; r < J->n_rows; r += J->nthreads) {
        long long flat = J->rows[r];
        long bh = (long)(flat / J->Nq); /* b*Hq + hq */
        long i = (long)(flat % J->Nq);
        long kvh = bh / group; /* b*Hkv + hq / (Hq/Hkv) */
        const double *kh = J->k + (size_t)kvh * J->Nk * J->D;
        const double *vh = J->v + (size_t)kvh * J->Nk * J->D;
        attend_row(J->q_rows + (size_t)r * J->D, kh, vh, i, J->Nk, J->D,
                   J->scale, J->causal, J->Nk - J->Nq, s,
                   J->o_rows + (size_t)r * J->D, J->lse_rows + r);
    }
    free(s);
    return NULL;
}

static int resolve_threads(int nthreads, long work)
{
    if (nthreads <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = n > 0 ? (int)n : 1;
    }
    if (nthreads > 256)
        nthreads = 256;
    if (work < nthreads)
        nthreads = work > 0 ? (int)work : 1;
    return nthreads;
}

/*
 * Attention for a chosen set of output rows.
 *   q_rows   [n_rows, D]   the query row of each selected output row
 *   rows     [n_rows]      flattened index (b*Hq + hq)*Nq + i of each row
 *   k, v     [B, Hkv, Nk, D]
 *   o_rows   [n_rows, D], lse_rows [n_rows]  (written)
 * Returns the number of threads used (> 0), or -1 on bad arguments (also a
 * causal call with Nq > Nk) or an allocation failure.  nthreads <= 0 means
 * one per online CPU.
 */
int oracle_attention_rows_kv(const double *q_rows, const long long *rows,
                             long n_rows, const double *k, const double *v,
                             double *o_rows, double *lse_rows, long B, long Hq,
                             long Hkv, long Nq, long Nk, long D, double scale,
                             int causal, int nthreads)
{
    if (n_rows < 0 || B < 0 || Hq < 1 || Hkv < 1 || Hq % Hkv || Nq < 1 ||
        Nk < 1 || D < 1 || (causal && Nq > Nk))
        return -1;
    for (long r = 0; r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= (long long)B * Hq * Nq)
            return -1;
    int T = resolve_threads(nthreads, n_rows);
    pthread_t th[256];
    job_t jobs[256];
    int failed = 0;
    for (int t = 0; t < T; ++t) {
        job_t J = {q_rows, rows, n_rows, k, v, o_rows, lse_rows, Hq, Hkv,
                   Nq, Nk, D, scale, causal, t, T, 0};
        jobs[t] = J;
    }
    int started = 0;
    for (int t = 1; t < T; ++t) {
        if (pthread_create(&th[t], NULL, run_rows, &jobs[t]) != 0)
            break;
        started = t;
    }
    /* rows of threads that could not start are run here */
    for (int t = started + 1; t < T; ++t)
        run_rows(&jobs[t]);
    run_rows(&jobs[0]);
    for (int t = 1; t <= started; ++t)
        pthread_join(th[t], NULL);
    for (int t = 0; t < T; ++t)
        failed |= jobs[t].failed;
    return failed ? -1 : T;
}

/*
 * Attention over every row: q, o [B, Hq, Nq, D]; k, v [B, Hkv, Nk, D];
 * lse [B, Hq, Nq].  Same return convention as oracle_attention_rows_kv.
 */
int oracle_attention_kv(const double *q, const double *k, const double *v,
                        double *o, double *lse, long B, long Hq, long Hkv,
                        long Nq, long Nk, long D, double scale, int causal,
                        int nthreads)
{
    long n_rows = B * Hq * Nq;
    long long *rows = (long long *)malloc(sizeof(long long) * (size_t)(n_rows > 0 ? n_rows : 1));
    if (!rows)
        return -1;
    for (long r = 0; r < n_rows; ++r)
        rows[r] = r;
    int rc = oracle_attention_rows_kv(q, rows, n_rows, k, v, o, lse, B, Hq,
                                      Hkv, Nq, Nk, D, scale, causal, nthreads);
    free(rows);
    return rc;
}

/* Square problems (Nq == Nk == N): the two entry points above with N twice. */
int oracle_attention_rows(const double *q_rows, const long long *rows,
                          long n_rows, const double *k, const double *v,
                          double *o_rows, double *lse_rows, long B, long Hq,
                          long Hkv, long N, long D, double scale, int causal,
                          int nthreads)
{
    return oracle_attention_rows_kv(q_rows, rows, n_rows, k, v, o_rows,
                                    lse_rows, B, Hq, Hkv, N, N, D, scale,
                                    causal, nthreads);
}

int oracle_attention(const double *q, const double *k, const double *v,
                     double *o, double *lse, long B, long Hq, long Hkv,
                     long N, long D, double scale, int causal, int nthreads)
{
    return oracle_attention_kv(q, k, v, o, lse, B, Hq, Hkv, N, N, D, scale,
                               causal, nthreads);
}
