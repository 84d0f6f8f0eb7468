/*
 * Oracle: exact scaled-dot-product attention in IEEE binary64.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code with the CUDA kernels.
 *
 * What it computes is the plain three-step definition of attention that
 * the FlashAttention pages start from ("FlashAttention 深度解析", first
 * part, section 2.3 "标准注意力的 IO 分析": S = Q K^T, P = softmax(S),
 * O = P V; "FlashAttention: как реально считается attention на GPU",
 * section "Куда утекает трафик: naive attention") with the scale applied
 * to the scores before the softmax, and the per-row log-sum-exp that the
 * FlashAttention-2 algorithm writes beside O ("04 Transformers, Attention,
 * and FlashAttention", Algorithm 1, steps 13 and 15: L_i = m_i + log l_i,
 * which equals logsumexp of the row).  For one query row i:
 *
 *     s_j   = scale * <q_i, k_j>         for every allowed key j
 *     M     = max_j s_j
 *     Z     = sum_j exp(s_j - M)
 *     o_i   = (sum_j exp(s_j - M) v_j) / Z
 *     lse_i = M + log Z
 *
 * Allowed keys are 0 <= j < L, or 0 <= j <= i with the causal mask
 * ("FlashAttention 深度解析", second part, section 2.3 "因果掩码优化":
 * query i attends to keys j <= i).  Subtracting M is the safe-softmax
 * rewrite of the same quantity (it cancels between numerator and
 * denominator), not an approximation.
 *
 * The score row is materialised one row at a time, so memory is O(L)
 * per thread, not O(L^2).  No blocking, fusion or reordering beyond that
 * definition: each sum runs over j in ascending order.  Threads (POSIX)
 * split the rows; each row is computed by one thread from start to end,
 * so the result does not depend on the thread count.
 *
 * Build: plain C11, -ffp-contract=off, no fast-math (see build.py).
 */
#include <math.h>
#include <pthread.h>
#include <stdatomic.h>
#include <stdint.h>
#include <stdlib.h>
#include <unistd.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_NOMEM 2

typedef struct {
    const double *q, *k, *v;
    int64_t n_heads, L, d;
    double scale;
    int causal;
    const int64_t *rows; /* NULL: every row in order */
    int64_t n_rows;
    double *o, *lse;
    atomic_llong next;   /* next unclaimed output index */
    atomic_int failed;
} job_t;

enum { ROWS_PER_CLAIM = 8 };

/* One query row: the five lines of the definition above. */
static void attention_row(const job_t *job, int64_t flat_row, double *s,
                          double *o_row, double *lse_out)
{
    const int64_t L = job->L, d = job->d;
    const int64_t head = flat_row / L;
    const int64_t i = flat_row % L;
    const double *qi = job->q + flat_row * d;
    const double *kh = job->k + head * L * d;
    const double *vh = job->v + head * L * d;
    const int64_t n_keys = job->causal ? i + 1 : L;

    /* s_j = scale * <q_i, k_j> */
    for (int64_t j = 0; j < n_keys; ++j) {
        const double *kj = kh + j * d;
        double dot = 0.0;
        for (int64_t t = 0; t < d; ++t)
            dot += qi[t] * kj[t];
        s[j] = job->scale * dot;
    }
    /* M = max_j s_j */
    double M = s[0];
    for (int64_t j = 1; j < n_keys; ++j)
        if (s[j] > M)
            M = s[j];
    /* Z = sum_j exp(s_j - M); numerator = sum_j exp(s_j - M) v_j */
    for (int64_t t = 0; t < d; ++t)
        o_row[t] = 0.0;
    double Z = 0.0;
    for (int64_t j = 0; j < n_keys; ++j) {
        const double p = exp(s[j] - M);
        const double *vj = vh + j * d;
        Z += p;
        for (int64_t t = 0; t < d; ++t)
            o_row[t] += p * vj[t];
    }
    /* o_i = numerator / Z ; lse_i = M + log Z */
    for (int64_t t = 0; t < d; ++t)
        o_row[t] /= Z;
    *lse_out = M + log(Z);
}

static void *worker(void *arg)
{
    job_t *job = (job_t *)arg;
    double *s = (double *)malloc((size_t)job->L * sizeof(double));
    if (!s) {
        atomic_store(&job->failed, 1);
        return NULL;
    }
    for (;;) {
        const int64_t lo = atomic_fetch_add(&job->next, ROWS_PER_CLAIM);
        if (lo >= job->n_rows)
            break;
        const int64_t hi = lo + ROWS_PER_CLAIM < job->n_rows ? lo + ROWS_PER_CLAIM : job->n_rows;
        for (int64_t r = lo; r < hi; ++r) {
            const int64_t flat = job->rows ? job->rows[r] : r;
            attention_row(job, flat, s, job->o + r * job->d, job->lse + r);
        }
    }
    free(s);
    return NULL;
}

/*
 * q, k, v : binary64 arrays [n_heads, L, d], row-major, contiguous.
 * rows    : optional list of n_rows flat query indices (head * L + i); when
 *           NULL every row is computed (n_rows must equal n_heads * L).
 * o       : [n_rows, d] output;  lse : [n_rows] output.
 * n_threads <= 0 uses every online host core.
 * Returns ORACLE_OK, ORACLE_ERR_ARG or ORACLE_ERR_NOMEM.
 */
int oracle_attention_fp64(const double *q, const double *k, const double *v,
                          int64_t n_heads, int64_t L, int64_t d, double scale,
                          int causal, const int64_t *rows, int64_t n_rows,
                          double *o, double *lse, int n_threads)
{
    if (!q || !k || !v || !o || !lse || n_heads <= 0 || L <= 0 || d <= 0 || n_rows < 0)
        return ORACLE_ERR_ARG;
    if (causal != 0 && causal != 1)
        return ORACLE_ERR_ARG;
    if (!rows && n_rows != n_heads * L)
        return ORACLE_ERR_ARG;
    if (rows)
        for (int64_t r = 0; r < n_rows; ++r)
            if (rows[r] < 0 || rows[r] >= n_heads * L)
                return ORACLE_ERR_ARG;
    if (n_rows == 0)
        return ORACLE_OK;

    job_t job;
    job.q = q; job.k = k; job.v = v;
    job.n_heads = n_heads; job.L = L; job.d = d;
    job.scale = scale; job.causal = causal;
    job.rows = rows; job.n_rows = n_rows;
    job.o = o; job.lse = lse;
    atomic_init(&job.next, 0);
    atomic_init(&job.failed, 0);

    long cores = sysconf(_SC_NPROCESSORS_ONLN);
    int nt = n_threads > 0 ? n_threads : (int)(cores > 0 ? cores : 1);
    const int64_t claims = (n_rows + ROWS_PER_CLAIM - 1) / ROWS_PER_CLAIM;
    if (nt > claims)
        nt = (int)claims;
    if (nt <= 1) {
        worker(&job);
    } else {
        pthread_t *tid = (pthread_t *)malloc((size_t)nt * sizeof(pthread_t));
        if (!tid)
            return ORACLE_ERR_NOMEM;
        int started = 0;
        for (; started < nt; ++started)
            if (pthread_create(&tid[started], NULL, worker, &job) != 0)
                break;
        if (started == 0)
            worker(&job);
        for (int t = 0; t < started; ++t)
            pthread_join(tid[t], NULL);
        free(tid);
    }
    return atomic_load(&job.failed) ? ORACLE_ERR_NOMEM : ORACLE_OK;
}

/*
 * The softmax probabilities of one query row, p_j = exp(s_j - M) / Z for
 * j < n_keys (n_keys = L, or i + 1 when causal); p_out has room for L
 * values and entries past n_keys are set to 0.  Same definition as above.
 */
int oracle_row_probs_fp64(const double *q, const double *k, int64_t L, int64_t d,
                          double scale, int causal, int64_t i, double *p_out)
{
    if (!q || !k || !p_out || L <= 0 || d <= 0 || i < 0 || i >= L)
        return ORACLE_ERR_ARG;
    const int64_t n_keys = causal ? i + 1 : L;
    const double *qi = q + i * d;
    for (int64_t j = 0; j < n_keys; ++j) {
        double dot = 0.0;
        for (int64_t t = 0; t < d; ++t)
            dot += qi[t] * k[j * d + t];
        p_out[j] = scale * dot;
    }
    double M = p_out[0];
    for (int64_t j = 1; j < n_keys; ++j)
        if (p_out[j] > M)
            M = p_out[j];
    double Z = 0.0;
    for (int64_t j = 0; j < n_keys; ++j) {
        p_out[j] = exp(p_out[j] - M);
        Z += p_out[j];
    }
    for (int64_t j = 0; j < n_keys; ++j)
        p_out[j] /= Z;
    for (int64_t j = n_keys; j < L; ++j)
        p_out[j] = 0.0;
    return ORACLE_OK;
}
