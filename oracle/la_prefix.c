/*
 * la_prefix.c -- the O(N D^2) prefix (recurrent-state) form of the same linear attention, in fp64.
 *
 * TEST INFRASTRUCTURE ONLY, like la_oracle.c, and independent of it: it shares no code with the
 * explicit form, so that the two can pin each other.  Its shape follows the running-state update
 * S <- S + k_t v_t^T printed on the cloud.baidu.com page (section 2, "state matrix recurrence"),
 * extended with the sums that the normalised kernel needs.  Per head, with rows i = 0..N-1:
 *
 *   S_i = sum_{j in J(i)} k_j v_j^T   z_i = sum_{j in J(i)} k_j   a_i = sum_{j in J(i)} v_j   n_i = |J(i)|
 *   J(i) = {0..i} when causal, all rows otherwise
 *   g_i  = c n_i + q_i . z_i            O_i = (c a_i + S_i^T q_i) / g_i
 *
 * and for the gradient of L = sum dO . O, with dOt_i = dO_i / g_i and dt_i = (dO_i . O_i) / g_i:
 *
 *   dQ_i = S_i dOt_i - dt_i z_i
 *   P_j  = sum_{i in I(j)} q_i dOt_i^T   y_j = sum_{i in I(j)} dt_i q_i   e_j = sum_{i in I(j)} dOt_i
 *   I(j) = {j..N-1} when causal, all rows otherwise
 *   dK_j = P_j v_j - y_j                 dV_j = c e_j + P_j^T k_j
 *
 * These follow from the explicit definitions by exchanging the order of summation; they are what the
 * pages' O(N D^2) time and O(N D) memory claims (sciencestack.ai page, TL;DR) rest on.
 */
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    const double *Q, *K, *V, *dO;
    long N, D;
    int causal;
    double c;
    double *O, *g, *dQ, *dK, *dV;
    long n_heads;
    int n_threads, tid, failed;
} prefix_job;

/* Forward over one head; st holds S (D*D), z (D), a (D). */
static void prefix_forward_head(const prefix_job *jb, long bh, double *st) {
    const long N = jb->N, D = jb->D, off = bh * N * D;
    const double *q = jb->Q + off, *k = jb->K + off, *v = jb->V + off;
    double *S = st, *z = st + D * D, *a = z + D;
    memset(st, 0, sizeof(double) * (size_t)(D * D + 2 * D));
    long n = 0;
    if (!jb->causal) {
        for (long j = 0; j < N; ++j) {
            for (long d = 0; d < D; ++d) {
                for (long e = 0; e < D; ++e) S[d * D + e] += k[j * D + d] * v[j * D + e];
                z[d] += k[j * D + d];
                a[d] += v[j * D + d];
            }
        }
        n = N;
    }
    for (long i = 0; i < N; ++i) {
        if (jb->causal) {
            for (long d = 0; d < D; ++d) {
                for (long e = 0; e < D; ++e) S[d * D + e] += k[i * D + d] * v[i * D + e];
                z[d] += k[i * D + d];
                a[d] += v[i * D + d];
            }
            n = i + 1;
        }
        double gi = jb->c * (double)n;
        for (long d = 0; d < D; ++d) gi += q[i * D + d] * z[d];
        jb->g[bh * N + i] = gi;
        for (long e = 0; e < D; ++e) {
            double num = jb->c * a[e];
            for (long d = 0; d < D; ++d) num += S[d * D + e] * q[i * D + d];
            jb->O[off + i * D + e] = num / gi;
        }
    }
}

/* Backward over one head; st holds S or P (D*D), z or y (D), a or e (D), then g[N] and dt[N]. */
static void prefix_backward_head(const prefix_job *jb, long bh, double *st) {
    const long N = jb->N, D = jb->D, off = bh * N * D;
    const double *q = jb->Q + off, *k = jb->K + off, *v = jb->V + off, *dO = jb->dO + off;
    double *dq = jb->dQ + off, *dk = jb->dK + off, *dv = jb->dV + off;
    double *S = st, *z = st + D * D, *a = z + D, *gv = a + D, *dt = gv + N;
    const double c = jb->c;

    /* forward-direction sweep: g_i, O_i (kept only as delta_i), dQ_i */
    memset(st, 0, sizeof(double) * (size_t)(D * D + 2 * D));
    long n = 0;
    if (!jb->causal) {
        for (long j = 0; j < N; ++j)
            for (long d = 0; d < D; ++d) {
                for (long e = 0; e < D; ++e) S[d * D + e] += k[j * D + d] * v[j * D + e];
                z[d] += k[j * D + d];
                a[d] += v[j * D + d];
            }
        n = N;
    }
    for (long i = 0; i < N; ++i) {
        if (jb->causal) {
            for (long d = 0; d < D; ++d) {
                for (long e = 0; e < D; ++e) S[d * D + e] += k[i * D + d] * v[i * D + e];
                z[d] += k[i * D + d];
                a[d] += v[i * D + d];
            }
            n = i + 1;
        }
        double gi = c * (double)n;
        for (long d = 0; d < D; ++d) gi += q[i * D + d] * z[d];
        double delta = 0.0;
        for (long e = 0; e < D; ++e) {
            double num = c * a[e];
            for (long d = 0; d < D; ++d) num += S[d * D + e] * q[i * D + d];
            delta += dO[i * D + e] * (num / gi);
        }
        gv[i] = gi;
        dt[i] = delta / gi;
        for (long d = 0; d < D; ++d) {
            double s = 0.0;
            for (long e = 0; e < D; ++e) s += S[d * D + e] * (dO[i * D + e] / gi);
            dq[i * D + d] = s - dt[i] * z[d];
        }
    }

    /* reverse sweep: P (in S), y (in z), e (in a) */
    double *P = S, *y = z, *ev = a;
    memset(st, 0, sizeof(double) * (size_t)(D * D + 2 * D));
    if (!jb->causal) {
        for (long i = 0; i < N; ++i)
            for (long d = 0; d < D; ++d) {
                for (long e = 0; e < D; ++e) P[d * D + e] += q[i * D + d] * (dO[i * D + e] / gv[i]);
                y[d] += dt[i] * q[i * D + d];
                ev[d] += dO[i * D + d] / gv[i];
            }
    }
    for (long j = N - 1; j >= 0; --j) {
        if (jb->causal) {
            for (long d = 0; d < D; ++d) {
                for (long e = 0; e < D; ++e) P[d * D + e] += q[j * D + d] * (dO[j * D + e] / gv[j]);
                y[d] += dt[j] * q[j * D + d];
                ev[d] += dO[j * D + d] / gv[j];
            }
        }
        for (long d = 0; d < D; ++d) {
            double s = 0.0;
            for (long e = 0; e < D; ++e) s += P[d * D + e] * v[j * D + e];
            dk[j * D + d] = s - y[d];
        }
        for (long e = 0; e < D; ++e) {
            double s = c * ev[e];
            for (long d = 0; d < D; ++d) s += P[d * D + e] * k[j * D + d];
            dv[j * D + e] = s;
        }
    }
}

static void *prefix_worker(void *p) {
    prefix_job *jb = (prefix_job *)p;
    long len = jb->D * jb->D + 2 * jb->D + 2 * jb->N;
    double *st = (double *)malloc(sizeof(double) * (size_t)len);
    if (!st) {
        jb->failed = 1;
        return NULL;
    }
    for (long bh = jb->tid; bh < jb->n_heads; bh += jb->n_threads) {
        if (jb->dQ)
            prefix_backward_head(jb, bh, st);
        else
            prefix_forward_head(jb, bh, st);
    }
    free(st);
    return NULL;
}

static int prefix_run(prefix_job proto) {
    int nt = proto.n_threads;
    if (nt <= 0) {
        long n = sysconf(_SC_NPROCESSORS_ONLN);
        nt = n > 0 ? (int)n : 1;
    }
    if (nt > proto.n_heads) nt = (int)proto.n_heads;
    if (nt < 1) return 0;
    prefix_job *jobs = (prefix_job *)calloc((size_t)nt, sizeof(prefix_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nt, sizeof(pthread_t));
    int *started = (int *)calloc((size_t)nt, sizeof(int));
    if (!jobs || !th || !started) {
        free(jobs);
        free(th);
        free(started);
        return -1;
    }
    for (int t = 0; t < nt; ++t) {
        jobs[t] = proto;
        jobs[t].n_threads = nt;
        jobs[t].tid = t;
        jobs[t].failed = 0;
        started[t] = t > 0 && pthread_create(&th[t], NULL, prefix_worker, &jobs[t]) == 0;
    }
    prefix_worker(&jobs[0]);
    for (int t = 1; t < nt; ++t) {
        if (started[t])
            pthread_join(th[t], NULL);
        else
            prefix_worker(&jobs[t]);
    }
    int rc = 0;
    for (int t = 0; t < nt; ++t) rc |= jobs[t].failed;
    free(jobs);
    free(th);
    free(started);
    return rc ? -1 : 0;
}

int la_prefix_forward(const double *Q, const double *K, const double *V, long B, long H, long N, long D, int causal,
                      double c, double *O, double *g, int n_threads) {
    if (B < 0 || H < 0 || N < 0 || D < 1) return -1;
    prefix_job jb = {Q, K, V, NULL, N, D, causal, c, O, g, NULL, NULL, NULL, B * H, n_threads, 0, 0};
    return prefix_run(jb);
}

int la_prefix_backward(const double *Q, const double *K, const double *V, const double *dO, long B, long H, long N,
                       long D, int causal, double c, double *dQ, double *dK, double *dV, int n_threads) {
    if (B < 0 || H < 0 || N < 0 || D < 1) return -1;
    prefix_job jb = {Q, K, V, dO, N, D, causal, c, NULL, NULL, dQ, dK, dV, B * H, n_threads, 0, 0};
    return prefix_run(jb);
}
