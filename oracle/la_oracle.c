/*
 * la_oracle.c -- explicit O(N^2 D) fp64 CPU oracle for normalised linear attention.
 *
 * TEST INFRASTRUCTURE ONLY.  The CUDA library never links, loads or calls this file.  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg use it.  It shares no code, header,
 * table or helper with the CUDA path.
 *
 * Source: "Transformer Based Linear Attention with Optimized GPU Kernel Implementation"
 * (A. Gerami, R. Duraiswami, arXiv 2510.21956).  The sciencestack.ai page (TL;DR) says that the
 * linear-attention (LA) head has a forward/backward formulation, a normalisation scheme, analytical
 * gradients, O(N D^2) time and O(N D) memory.  The shd-paper.top page (abstract) gives the setting:
 * N tokens, each embedded in a D-dimensional head.  No page prints the formula.  This file implements
 * the reading that the rest of the pages support (normalised linear kernel with constant c):
 *
 *   W_ij = m_ij (c + q_i . k_j)      m_ij = [j <= i] when causal, else 1;  c = 1 in the library
 *   g_i  = sum_j W_ij                the normaliser (the "normalization scheme")
 *   A_ij = W_ij / g_i                normalised weights; each row sums to one
 *   O_i  = sum_j A_ij v_j
 *
 * and, for the backward ("analytical gradients ... for the LA head"), the exact gradient of the
 * scalar L = sum_i dO_i . O_i, taken by the chain rule through the division by g_i:
 *
 *   delta_i = dO_i . O_i
 *   dW_ij   = m_ij (dO_i . v_j - delta_i) / g_i
 *   dQ_i    = sum_j dW_ij k_j       dK_j = sum_i dW_ij q_i       dV_j = sum_i A_ij dO_i
 *
 * Everything is fp64, loops run in index order, and no step is blocked, fused or reordered: the N x N
 * weights are formed one row at a time, exactly as written above.  Tensors are contiguous
 * [B, H, N, D] (row i of head (b, h) at ((b H + h) N + i) D); the normaliser is [B, H, N].
 */
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ---------------------------------------------------------------- threading (plain pthreads) --- */

typedef void (*oracle_item_fn)(long item, void *ctx, double *scratch);

typedef struct {
    oracle_item_fn fn;
    void *ctx;
    long n_items;
    long scratch_len;
    int n_threads;
    int tid;
    int failed;
} oracle_job;

static void *oracle_worker(void *p) {
    oracle_job *job = (oracle_job *)p;
    double *scratch = (double *)malloc(sizeof(double) * (size_t)(job->scratch_len > 0 ? job->scratch_len : 1));
    if (!scratch) {
        job->failed = 1;
        return NULL;
    }
    for (long it = job->tid; it < job->n_items; it += job->n_threads) job->fn(it, job->ctx, scratch);
    free(scratch);
    return NULL;
}

static int oracle_threads(int requested) {
    if (requested > 0) return requested;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/* Runs fn(item) for item in [0, n_items) on up to n_threads threads, each with its own scratch. */
static int oracle_parallel(oracle_item_fn fn, void *ctx, long n_items, long scratch_len, int n_threads) {
    int nt = oracle_threads(n_threads);
    if (nt > n_items) nt = (int)(n_items > 0 ? n_items : 1);
    oracle_job *jobs = (oracle_job *)calloc((size_t)nt, sizeof(oracle_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nt, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return -1;
    }
    int rc = 0;
    for (int t = 0; t < nt; ++t) {
        jobs[t] = (oracle_job){fn, ctx, n_items, scratch_len, nt, t, 0};
        if (t > 0 && pthread_create(&th[t], NULL, oracle_worker, &jobs[t]) != 0) {
            jobs[t].failed = 2; /* run it inline below instead */
        }
    }
    oracle_worker(&jobs[0]);
    for (int t = 1; t < nt; ++t) {
        if (jobs[t].failed == 2) {
            jobs[t].failed = 0;
            oracle_worker(&jobs[t]);
        } else {
            pthread_join(th[t], NULL);
        }
    }
    for (int t = 0; t < nt; ++t) rc |= jobs[t].failed;
    free(jobs);
    free(th);
    return rc ? -1 : 0;
}

/* ------------------------------------------------------------------------- shared arguments --- */

typedef struct {
    const double *Q, *K, *V, *dO;
    long B, H, N, D;
    int causal;
    double c;
    double *O, *g;            /* forward outputs */
    double *dQ, *dK, *dV;     /* backward outputs */
    const long *rows;         /* flat (b H + h) N + i indices, for the sampled-row entry points */
    long n_rows;
} oracle_args;

static double dot(const double *x, const double *y, long D) {
    double s = 0.0;
    for (long d = 0; d < D; ++d) s += x[d] * y[d];
    return s;
}

/* Row i of one head: fills w[j] = W_ij for the unmasked j (j < jend) and returns g_i = sum_j W_ij. */
static double weights_row(const double *q, const double *k, long i, long N, long D, int causal, double c,
                          double *w, long *jend_out) {
    long jend = causal ? i + 1 : N;
    double gi = 0.0;
    for (long j = 0; j < jend; ++j) {
        w[j] = c + dot(q + i * D, k + j * D, D); /* W_ij = m_ij (c + q_i . k_j), m_ij = 1 here */
        gi += w[j];                              /* g_i = sum_j W_ij */
    }
    *jend_out = jend;
    return gi;
}

/* O_i = sum_j (W_ij / g_i) v_j for the row whose weights are in w. */
static void output_row(const double *w, long jend, double gi, const double *v, long D, double *o) {
    for (long d = 0; d < D; ++d) o[d] = 0.0;
    for (long j = 0; j < jend; ++j) {
        double a = w[j] / gi; /* A_ij */
        for (long d = 0; d < D; ++d) o[d] += a * v[j * D + d];
    }
}

/* ------------------------------------------------------------------------------- forward --- */

static void forward_head(long bh, void *ctx, double *w) {
    const oracle_args *a = (const oracle_args *)ctx;
    const long N = a->N, D = a->D, off = bh * N * D;
    const double *q = a->Q + off, *k = a->K + off, *v = a->V + off;
    for (long i = 0; i < N; ++i) {
        long jend;
        double gi = weights_row(q, k, i, N, D, a->causal, a->c, w, &jend);
        a->g[bh * N + i] = gi;
        output_row(w, jend, gi, v, D, a->O + off + i * D);
    }
}

/* Full explicit forward: O [B,H,N,D] and the normaliser g [B,H,N]. */
int la_oracle_forward(const double *Q, const double *K, const double *V, long B, long H, long N, long D,
                      int causal, double c, double *O, double *g, int n_threads) {
    if (B < 0 || H < 0 || N < 0 || D < 1) return -1;
    if (B * H * N == 0) return 0;
    oracle_args a = {Q, K, V, NULL, B, H, N, D, causal, c, O, g, NULL, NULL, NULL, NULL, 0};
    return oracle_parallel(forward_head, &a, B * H, N, n_threads);
}

/* The normalised weights A (N x N, row-major, zeros where masked) of a single head. */
int la_oracle_weights(const double *q, const double *k, long N, long D, int causal, double c, double *A) {
    if (N < 0 || D < 1) return -1;
    double *w = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    if (!w) return -1;
    for (long i = 0; i < N; ++i) {
        long jend;
        double gi = weights_row(q, k, i, N, D, causal, c, w, &jend);
        for (long j = 0; j < N; ++j) A[i * N + j] = j < jend ? w[j] / gi : 0.0;
    }
    free(w);
    return 0;
}

/* Sampled rows: O_i and g_i for each flat row index in rows[] (cost O(N D) per row). */
static void forward_sampled_row(long r, void *ctx, double *w) {
    const oracle_args *a = (const oracle_args *)ctx;
    const long N = a->N, D = a->D;
    long flat = a->rows[r], bh = flat / N, i = flat % N, off = bh * N * D;
    long jend;
    double gi = weights_row(a->Q + off, a->K + off, i, N, D, a->causal, a->c, w, &jend);
    a->g[r] = gi;
    output_row(w, jend, gi, a->V + off, D, a->O + r * D);
}

int la_oracle_forward_rows(const double *Q, const double *K, const double *V, long B, long H, long N, long D,
                           int causal, double c, const long *rows, long n_rows, double *O_rows, double *g_rows,
                           int n_threads) {
    if (D < 1 || N < 1) return -1;
    for (long r = 0; r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= B * H * N) return -1;
    if (n_rows == 0) return 0;
    oracle_args a = {Q, K, V, NULL, B, H, N, D, causal, c, O_rows, g_rows, NULL, NULL, NULL, rows, n_rows};
    return oracle_parallel(forward_sampled_row, &a, n_rows, N, n_threads);
}

/* ------------------------------------------------------------------------------ backward --- */

/* scratch: w[N] then o[D] */
static void backward_head(long bh, void *ctx, double *scratch) {
    const oracle_args *a = (const oracle_args *)ctx;
    const long N = a->N, D = a->D, off = bh * N * D;
    const double *q = a->Q + off, *k = a->K + off, *v = a->V + off, *dO = a->dO + off;
    double *dq = a->dQ + off, *dk = a->dK + off, *dv = a->dV + off;
    double *w = scratch, *o = scratch + N;
    memset(dq, 0, sizeof(double) * (size_t)(N * D));
    memset(dk, 0, sizeof(double) * (size_t)(N * D));
    memset(dv, 0, sizeof(double) * (size_t)(N * D));
    for (long i = 0; i < N; ++i) {
        long jend;
        double gi = weights_row(q, k, i, N, D, a->causal, a->c, w, &jend); /* steps 1-2 */
        output_row(w, jend, gi, v, D, o);                                  /* steps 3-4 */
        double delta = dot(dO + i * D, o, D);                              /* delta_i = dO_i . O_i */
        for (long j = 0; j < jend; ++j) {
            double Aij = w[j] / gi;
            double dW = (dot(dO + i * D, v + j * D, D) - delta) / gi; /* dW_ij */
            for (long d = 0; d < D; ++d) {
                dq[i * D + d] += dW * k[j * D + d]; /* dQ_i = sum_j dW_ij k_j */
                dk[j * D + d] += dW * q[i * D + d]; /* dK_j = sum_i dW_ij q_i */
                dv[j * D + d] += Aij * dO[i * D + d]; /* dV_j = sum_i A_ij dO_i */
            }
        }
    }
}

/* Full explicit backward: dQ, dK, dV [B,H,N,D] of L = sum dO . O, with O recomputed in fp64. */
int la_oracle_backward(const double *Q, const double *K, const double *V, const double *dO, long B, long H,
                       long N, long D, int causal, double c, double *dQ, double *dK, double *dV, int n_threads) {
    if (B < 0 || H < 0 || N < 0 || D < 1) return -1;
    if (B * H * N == 0) return 0;
    oracle_args a = {Q, K, V, dO, B, H, N, D, causal, c, NULL, NULL, dQ, dK, dV, NULL, 0};
    return oracle_parallel(backward_head, &a, B * H, N + D, n_threads);
}

/* Sampled rows of dQ: dQ_i = sum_j dW_ij k_j needs only row i (cost O(N D)). scratch: w[N], o[D]. */
static void dq_sampled_row(long r, void *ctx, double *scratch) {
    const oracle_args *a = (const oracle_args *)ctx;
    const long N = a->N, D = a->D;
    long flat = a->rows[r], bh = flat / N, i = flat % N, off = bh * N * D;
    const double *q = a->Q + off, *k = a->K + off, *v = a->V + off, *dO = a->dO + off;
    double *w = scratch, *o = scratch + N, *dq = a->dQ + r * D;
    long jend;
    double gi = weights_row(q, k, i, N, D, a->causal, a->c, w, &jend);
    output_row(w, jend, gi, v, D, o);
    double delta = dot(dO + i * D, o, D);
    for (long d = 0; d < D; ++d) dq[d] = 0.0;
    for (long j = 0; j < jend; ++j) {
        double dW = (dot(dO + i * D, v + j * D, D) - delta) / gi;
        for (long d = 0; d < D; ++d) dq[d] += dW * k[j * D + d];
    }
}

int la_oracle_dq_rows(const double *Q, const double *K, const double *V, const double *dO, long B, long H, long N,
                      long D, int causal, double c, const long *rows, long n_rows, double *dQ_rows, int n_threads) {
    if (D < 1 || N < 1) return -1;
    for (long r = 0; r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= B * H * N) return -1;
    if (n_rows == 0) return 0;
    oracle_args a = {Q, K, V, dO, B, H, N, D, causal, c, NULL, NULL, dQ_rows, NULL, NULL, rows, n_rows};
    return oracle_parallel(dq_sampled_row, &a, n_rows, N + D, n_threads);
}

/*
 * Sampled rows of dK and dV: dK_j = sum_i dW_ij q_i and dV_j = sum_i A_ij dO_i run over every row i
 * that sees j (i >= j when causal, all i otherwise).  Each such row needs its own g_i and delta_i, so
 * this costs O((N - j) N D) per sampled j: cheap for j near the end of a causal head.
 * scratch: w[N], o[D].
 */
static void dkdv_sampled_row(long r, void *ctx, double *scratch) {
    const oracle_args *a = (const oracle_args *)ctx;
    const long N = a->N, D = a->D;
    long flat = a->rows[r], bh = flat / N, j = flat % N, off = bh * N * D;
    const double *q = a->Q + off, *k = a->K + off, *v = a->V + off, *dO = a->dO + off;
    double *w = scratch, *o = scratch + N, *dk = a->dK + r * D, *dv = a->dV + r * D;
    for (long d = 0; d < D; ++d) dk[d] = dv[d] = 0.0;
    for (long i = a->causal ? j : 0; i < N; ++i) {
        long jend;
        double gi = weights_row(q, k, i, N, D, a->causal, a->c, w, &jend);
        output_row(w, jend, gi, v, D, o);
        double delta = dot(dO + i * D, o, D);
        double Aij = w[j] / gi;
        double dW = (dot(dO + i * D, v + j * D, D) - delta) / gi;
        for (long d = 0; d < D; ++d) {
            dk[d] += dW * q[i * D + d];
            dv[d] += Aij * dO[i * D + d];
        }
    }
}

int la_oracle_dkdv_rows(const double *Q, const double *K, const double *V, const double *dO, long B, long H,
                        long N, long D, int causal, double c, const long *rows, long n_rows, double *dK_rows,
                        double *dV_rows, int n_threads) {
    if (D < 1 || N < 1) return -1;
    for (long r = 0; r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= B * H * N) return -1;
    if (n_rows == 0) return 0;
    oracle_args a = {Q, K, V, dO, B, H, N, D, causal, c, NULL, NULL, NULL, dK_rows, dV_rows, rows, n_rows};
    return oracle_parallel(dkdv_sampled_row, &a, n_rows, N + D, n_threads);
}
