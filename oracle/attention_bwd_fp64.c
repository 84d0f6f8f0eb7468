/*
 * Oracle: gradients of exact scaled-dot-product attention in IEEE binary64.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only the tests and the benchmark's CPU legs do.  It
 * shares no code with the CUDA kernels.
 *
 * What it computes.  Given Q, K, V, the output gradient dO and the forward
 * definition O = softmax(scale * Q K^T) V (with the causal mask when asked),
 * the gradients dQ, dK, dV of any loss whose gradient with respect to O is
 * dO.  The backward formulas are those of "FlashAttention 深度解析", first
 * part, section 4.1 (反向传播与显存优化 / 问题：注意力矩阵不被存储):
 *
 *     dV  = P^T dO
 *     dP  = dO V^T
 *     dS  = dP (.) P  -  P (.) rowsum(dP (.) P)
 *
 * where S are the scaled scores and P the softmax probabilities.  The
 * scores are S = scale * Q K^T, so the chain rule through that product gives
 *
 *     dQ = scale * dS K          dK = scale * dS^T Q .
 *
 * P is recomputed from the scores and the row statistics of the forward
 * pass (section 4.2, 重计算策略: P_ij = exp(S_ij - m_i) / l_i), never
 * stored as a matrix.  Masked (key > query) entries have P = 0 and no
 * gradient.
 *
 * Structure: three passes, each one of the lines above written out with
 * sums in ascending index order.
 *
 *   pass 1, per query row i:  s_ij = scale <q_i, k_j>, M_i = max_j s_ij,
 *            Z_i = sum_j exp(s_ij - M_i), P_ij = exp(s_ij - M_i) / Z_i,
 *            dP_ij = <dO_i, v_j>, c_i = sum_j dP_ij P_ij  (the row sum).
 *   pass 2, per key row j:    dV_j = sum_i P_ij dO_i,
 *                             dK_j = scale * sum_i dS_ij q_i,
 *            with dS_ij = P_ij (dP_ij - c_i), over the queries i that see j.
 *   pass 3, per query row i:  dQ_i = scale * sum_j dS_ij k_j.
 *
 * Passes 2 and 3 can be restricted to chosen rows, so that single rows of
 * a large problem are affordable; pass 1 then runs over every query row of
 * each head that has a chosen key row, plus the chosen query rows.  Threads
 * (POSIX) split the rows of each pass; every output row is computed by one
 * thread from start to end, so the result does not depend on the thread
 * count.
 *
 * Build: plain C11, -ffp-contract=off, no fast-math (see build.py).
 */
#include <math.h>
#include <pthread.h>
#include <stdatomic.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_NOMEM 2

typedef struct {
    const double *q, *k, *v, *dout;
    int64_t n_heads, L, d;
    double scale;
    int causal;
    /* row statistics of pass 1, [n_heads * L] each */
    double *M, *Z, *c;
    /* the work list of the current pass */
    const int64_t *items;
    int64_t n_items;
    int pass;
    double *out_a, *out_b; /* pass 2: dk, dv;  pass 3: dq */
    atomic_llong next;
    atomic_int failed;
} bwd_job_t;

enum { ITEMS_PER_CLAIM = 4 };

static double dot(const double *a, const double *b, int64_t d)
{
    double s = 0.0;
    for (int64_t t = 0; t < d; ++t)
        s += a[t] * b[t];
    return s;
}

/* Pass 1 for query row i of a head: M_i, Z_i and c_i. */
static void row_stats(const bwd_job_t *job, int64_t flat, double *s)
{
    const int64_t L = job->L, d = job->d;
    const int64_t head = flat / L, i = flat % L;
    const double *qi = job->q + flat * d;
    const double *doi = job->dout + flat * d;
    const double *kh = job->k + head * L * d;
    const double *vh = job->v + head * L * d;
    const int64_t n_keys = job->causal ? i + 1 : L;

    for (int64_t j = 0; j < n_keys; ++j)
        s[j] = job->scale * dot(qi, kh + j * d, d);
    double M = s[0];
    for (int64_t j = 1; j < n_keys; ++j)
        if (s[j] > M)
            M = s[j];
    double Z = 0.0;
    for (int64_t j = 0; j < n_keys; ++j)
        Z += exp(s[j] - M);
    double c = 0.0;
    for (int64_t j = 0; j < n_keys; ++j) {
        const double P = exp(s[j] - M) / Z;
        const double dP = dot(doi, vh + j * d, d);
        c += dP * P;
    }
    job->M[flat] = M;
    job->Z[flat] = Z;
    job->c[flat] = c;
}

/* P_ij and dS_ij of one (query i, key j) pair of a head, from pass 1. */
static void prob_and_grad(const bwd_job_t *job, int64_t head, int64_t i, int64_t j,
                          double *P_out, double *dS_out)
{
    const int64_t L = job->L, d = job->d;
    const int64_t fi = head * L + i, fj = head * L + j;
    const double s = job->scale * dot(job->q + fi * d, job->k + fj * d, d);
    const double P = exp(s - job->M[fi]) / job->Z[fi];
    const double dP = dot(job->dout + fi * d, job->v + fj * d, d);
    *P_out = P;
    *dS_out = P * (dP - job->c[fi]);
}

/* Pass 2 for key row j: dK_j and dV_j over the queries that see key j. */
static void key_grads(const bwd_job_t *job, int64_t flat, double *dk, double *dv)
{
    const int64_t L = job->L, d = job->d;
    const int64_t head = flat / L, j = flat % L;
    for (int64_t t = 0; t < d; ++t)
        dk[t] = dv[t] = 0.0;
    for (int64_t i = job->causal ? j : 0; i < L; ++i) {
        double P, dS;
        prob_and_grad(job, head, i, j, &P, &dS);
        const double *qi = job->q + (head * L + i) * d;
        const double *doi = job->dout + (head * L + i) * d;
        for (int64_t t = 0; t < d; ++t) {
            dv[t] += P * doi[t];
            dk[t] += dS * qi[t];
        }
    }
    for (int64_t t = 0; t < d; ++t)
        dk[t] *= job->scale;
}

/* Pass 3 for query row i: dQ_i over the keys that query i sees. */
static void query_grad(const bwd_job_t *job, int64_t flat, double *dq)
{
    const int64_t L = job->L, d = job->d;
    const int64_t head = flat / L, i = flat % L;
    const int64_t n_keys = job->causal ? i + 1 : L;
    for (int64_t t = 0; t < d; ++t)
        dq[t] = 0.0;
    for (int64_t j = 0; j < n_keys; ++j) {
        double P, dS;
        prob_and_grad(job, head, i, j, &P, &dS);
        const double *kj = job->k + (head * L + j) * d;
        for (int64_t t = 0; t < d; ++t)
            dq[t] += dS * kj[t];
    }
    for (int64_t t = 0; t < d; ++t)
        dq[t] *= job->scale;
}

static void *bwd_worker(void *arg)
{
    bwd_job_t *job = (bwd_job_t *)arg;
    double *s = NULL;
    if (job->pass == 1) {
        s = (double *)malloc((size_t)job->L * sizeof(double));
        if (!s) {
            atomic_store(&job->failed, 1);
            return NULL;
        }
    }
    for (;;) {
        const int64_t lo = atomic_fetch_add(&job->next, ITEMS_PER_CLAIM);
        if (lo >= job->n_items)
            break;
        const int64_t hi = lo + ITEMS_PER_CLAIM < job->n_items ? lo + ITEMS_PER_CLAIM : job->n_items;
        for (int64_t r = lo; r < hi; ++r) {
            const int64_t flat = job->items[r];
            if (job->pass == 1)
                row_stats(job, flat, s);
            else if (job->pass == 2)
                key_grads(job, flat, job->out_a + r * job->d, job->out_b + r * job->d);
            else
                query_grad(job, flat, job->out_a + r * job->d);
        }
    }
    free(s);
    return NULL;
}

static int run_pass(bwd_job_t *job, int pass, const int64_t *items, int64_t n_items,
                    double *out_a, double *out_b, int n_threads)
{
    if (n_items == 0)
        return ORACLE_OK;
    job->pass = pass;
    job->items = items;
    job->n_items = n_items;
    job->out_a = out_a;
    job->out_b = out_b;
    atomic_store(&job->next, 0);
    long cores = sysconf(_SC_NPROCESSORS_ONLN);
    int nt = n_threads > 0 ? n_threads : (int)(cores > 0 ? cores : 1);
    const int64_t claims = (n_items + ITEMS_PER_CLAIM - 1) / ITEMS_PER_CLAIM;
    if (nt > claims)
        nt = (int)claims;
    if (nt <= 1) {
        bwd_worker(job);
    } else {
        pthread_t *tid = (pthread_t *)malloc((size_t)nt * sizeof(pthread_t));
        if (!tid)
            return ORACLE_ERR_NOMEM;
        int started = 0;
        for (; started < nt; ++started)
            if (pthread_create(&tid[started], NULL, bwd_worker, job) != 0)
                break;
        if (started == 0)
            bwd_worker(job);
        for (int t = 0; t < started; ++t)
            pthread_join(tid[t], NULL);
        free(tid);
    }
    return atomic_load(&job->failed) ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/*
 * q, k, v, dout : binary64 arrays [n_heads, L, d], row-major, contiguous.
 * key_rows      : n_key_rows flat key indices (head * L + j) whose dK and dV
 *                 rows are wanted, or NULL for every key (n_key_rows must
 *                 then be n_heads * L).
 * query_rows    : likewise for the dQ rows.
 * dq            : [n_query_rows, d];  dk, dv : [n_key_rows, d].
 * n_threads <= 0 uses every online host core.
 * Returns ORACLE_OK, ORACLE_ERR_ARG or ORACLE_ERR_NOMEM.
 */
int oracle_attention_bwd_fp64(const double *q, const double *k, const double *v,
                              const double *dout, int64_t n_heads, int64_t L, int64_t d,
                              double scale, int causal, const int64_t *key_rows,
                              int64_t n_key_rows, const int64_t *query_rows,
                              int64_t n_query_rows, double *dq, double *dk, double *dv,
                              int n_threads)
{
    if (!q || !k || !v || !dout || n_heads <= 0 || L <= 0 || d <= 0)
        return ORACLE_ERR_ARG;
    if (causal != 0 && causal != 1)
        return ORACLE_ERR_ARG;
    if (n_key_rows < 0 || n_query_rows < 0)
        return ORACLE_ERR_ARG;
    const int64_t n_flat = n_heads * L;
    if ((!key_rows && n_key_rows != n_flat) || (!query_rows && n_query_rows != n_flat))
        return ORACLE_ERR_ARG;
    if ((n_key_rows > 0 && (!dk || !dv)) || (n_query_rows > 0 && !dq))
        return ORACLE_ERR_ARG;
    for (int64_t r = 0; key_rows && r < n_key_rows; ++r)
        if (key_rows[r] < 0 || key_rows[r] >= n_flat)
            return ORACLE_ERR_ARG;
    for (int64_t r = 0; query_rows && r < n_query_rows; ++r)
        if (query_rows[r] < 0 || query_rows[r] >= n_flat)
            return ORACLE_ERR_ARG;

    int rc = ORACLE_ERR_NOMEM;
    double *stats = (double *)malloc((size_t)n_flat * 3 * sizeof(double));
    unsigned char *need = (unsigned char *)calloc((size_t)n_flat, 1);
    unsigned char *head_needed = (unsigned char *)calloc((size_t)n_heads, 1);
    int64_t *items = (int64_t *)malloc((size_t)(n_flat > n_key_rows ? n_flat : n_key_rows) *
                                           sizeof(int64_t) +
                                       (size_t)n_query_rows * sizeof(int64_t) + 8);
    if (!stats || !need || !head_needed || !items)
        goto done;

    bwd_job_t job;
    memset(&job, 0, sizeof(job));
    job.q = q; job.k = k; job.v = v; job.dout = dout;
    job.n_heads = n_heads; job.L = L; job.d = d;
    job.scale = scale; job.causal = causal;
    job.M = stats; job.Z = stats + n_flat; job.c = stats + 2 * n_flat;
    atomic_init(&job.next, 0);
    atomic_init(&job.failed, 0);

    /* pass 1 runs over every query row of a head with a wanted key row
       (any key's gradient sums over all queries), plus the wanted dQ rows */
    for (int64_t r = 0; r < n_key_rows; ++r)
        head_needed[(key_rows ? key_rows[r] : r) / L] = 1;
    for (int64_t h = 0; h < n_heads; ++h)
        if (head_needed[h])
            memset(need + h * L, 1, (size_t)L);
    for (int64_t r = 0; r < n_query_rows; ++r)
        need[query_rows ? query_rows[r] : r] = 1;
    int64_t n1 = 0;
    for (int64_t f = 0; f < n_flat; ++f)
        if (need[f])
            items[n1++] = f;
    rc = run_pass(&job, 1, items, n1, NULL, NULL, n_threads);
    if (rc != ORACLE_OK)
        goto done;

    for (int64_t r = 0; r < n_key_rows; ++r)
        items[r] = key_rows ? key_rows[r] : r;
    rc = run_pass(&job, 2, items, n_key_rows, dk, dv, n_threads);
    if (rc != ORACLE_OK)
        goto done;

    for (int64_t r = 0; r < n_query_rows; ++r)
        items[r] = query_rows ? query_rows[r] : r;
    rc = run_pass(&job, 3, items, n_query_rows, dq, NULL, n_threads);

done:
    free(stats);
    free(need);
    free(head_needed);
    free(items);
    return rc;
}
