/*
 * Float64 CPU oracle for exact scaled-dot-product attention, forward and
 * backward.  TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load it; the product path never does.  It shares
 * no code, header or constant with the CUDA library.
 *
 * What it computes (the plain definition, not the tiled algorithm):
 *
 *   Forward, per head and per query row i
 *   ("FlashAttention: Move Less, Not Compute Less", section "The Multiplication
 *   May Not Be the Slow Part": S = QK^T, P = softmax(S), O = PV; the 1/sqrt(d)
 *   factor and the causal rule "query i sees keys 0..i" from the course page
 *   "10 FlashAttention", sections 1 and 4):
 *     s_j  = scale * sum_c Q[i,c] K[j,c]          for j in allowed(i)
 *     m    = max_j s_j
 *     l    = sum_j exp(s_j - m)                    (stable softmax, section
 *            "Tiling Is Easy; Softmax Couples the Entire Row" of the same essay)
 *     P_j  = exp(s_j - m) / l
 *     O[i] = sum_j P_j V[j]
 *     L[i] = m + ln(l)    (the per-row log-sum-exp kept for the backward pass,
 *            "FlashAttention-2: Why the Attention Bottleneck Wasn't Where Everyone
 *            Was Looking", section "FA2 change #1: Stop dividing so much")
 *   allowed(i) = {0..N-1}, or {0..i} when causal.  Masked keys are left out of
 *   every sum, which is what adding -inf to their scores means.
 *
 *   Decode (course page "10 FlashAttention", section "The decode variant:
 *   FlashDecoding": a few query rows per sequence against a long key/value cache):
 *   the same per-row definition with Nq query rows and Nk keys per head and no
 *   mask, allowed(i) = {0..Nk-1}.  How the GPU splits the keys and merges the
 *   partial results is not the oracle's business; it computes each row whole.
 *
 *   Backward (the pages only say that S and P are rebuilt from the saved
 *   statistics; the formulas are the chain rule applied to the forward above):
 *     dP_j  = dO[i] . V[j]
 *     D_i   = sum_j P_j dP_j
 *     dS_j  = P_j (dP_j - D_i)
 *     dQ[i] = scale * sum_j dS_j K[j]
 *     dK[j] += scale * dS_j Q[i]
 *     dV[j] += P_j dO[i]
 *
 * Every full score row of length N is built; nothing is blocked, fused or
 * reordered.  Tensors are contiguous [BH][N][d] float64.  Work is split over
 * rows with POSIX threads; each row is computed by one thread in a fixed order,
 * so the forward result does not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const double *q, *k, *v, *dout;
    double *o, *lse, *dq, *dk, *dv;
    long BH, N, d;
    long Nq;          /* decode: query rows per head (N is then the key count) */
    int causal;
    double scale;
    const long *rows; /* NULL: every row; else the rows to compute in each head */
    long nrows;
    long bh;          /* backward: the head being processed */
    long row_begin, row_end;
    double *dk_part, *dv_part; /* backward: this thread's partial dK, dV of head bh */
} job_t;

static long n_allowed(long i, long N, int causal) { return causal ? i + 1 : N; }

/* Scores, max, exponentials and sum of one query row; returns m, writes l. */
static double score_row(const double *qi, const double *K, long n, long d, double scale,
                        double *s, double *l_out) {
    double m = -INFINITY;
    for (long j = 0; j < n; ++j) {
        const double *kj = K + j * d;
        double acc = 0.0;
        for (long c = 0; c < d; ++c) acc += qi[c] * kj[c];
        s[j] = scale * acc;
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (long j = 0; j < n; ++j) {
        s[j] = exp(s[j] - m);
        l += s[j];
    }
    *l_out = l;
    return m;
}

/* O row and L of query row i of one head; s is scratch of length N. */
static void forward_row(const double *Q, const double *K, const double *V, long N, long d,
                        long i, int causal, double scale, double *s, double *o_i,
                        double *lse_i) {
    long n = n_allowed(i, N, causal);
    double l;
    double m = score_row(Q + i * d, K, n, d, scale, s, &l);
    for (long c = 0; c < d; ++c) o_i[c] = 0.0;
    for (long j = 0; j < n; ++j) {
        double p = s[j] / l;
        const double *vj = V + j * d;
        for (long c = 0; c < d; ++c) o_i[c] += p * vj[c];
    }
    *lse_i = m + log(l);
}

static void *fwd_worker(void *arg) {
    job_t *jb = (job_t *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)(jb->N > 0 ? jb->N : 1));
    long per_head = jb->rows ? jb->nrows : jb->N;
    for (long t = jb->row_begin; t < jb->row_end; ++t) {
        long bh = t / per_head, r = t % per_head;
        long i = jb->rows ? jb->rows[r] : r;
        size_t head = (size_t)bh * (size_t)jb->N * (size_t)jb->d;
        forward_row(jb->q + head, jb->k + head, jb->v + head, jb->N, jb->d, i, jb->causal,
                    jb->scale, s, jb->o + (size_t)t * (size_t)jb->d, jb->lse + t);
    }
    free(s);
    return NULL;
}

/* Decode rows: t = bh * Nq + i; q, o are [BH][Nq][d], k, v are [BH][N][d]. */
static void *dec_worker(void *arg) {
    job_t *jb = (job_t *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)(jb->N > 0 ? jb->N : 1));
    for (long t = jb->row_begin; t < jb->row_end; ++t) {
        long bh = t / jb->Nq, i = t % jb->Nq;
        const double *Q = jb->q + (size_t)bh * (size_t)jb->Nq * (size_t)jb->d;
        size_t kv = (size_t)bh * (size_t)jb->N * (size_t)jb->d;
        forward_row(Q, jb->k + kv, jb->v + kv, jb->N, jb->d, i, 0, jb->scale, s,
                    jb->o + (size_t)t * (size_t)jb->d, jb->lse + t);
    }
    free(s);
    return NULL;
}

static int run_threads(job_t *base, long total, int nthreads, void *(*fn)(void *),
                       job_t *jobs) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > total) nthreads = (int)(total > 0 ? total : 1);
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!th) return -1;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = *base;
        jobs[t].row_begin = base->row_begin + total * t / nthreads;
        jobs[t].row_end = base->row_begin + total * (t + 1) / nthreads;
        if (pthread_create(&th[t], NULL, fn, &jobs[t]) != 0) {
            for (int u = 0; u < t; ++u) pthread_join(th[u], NULL);
            free(th);
            return -1;
        }
    }
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    free(th);
    return 0;
}

/* Forward over every row.  o: [BH][N][d], lse: [BH][N].  Returns 0 on success. */
int oracle_fwd(const double *q, const double *k, const double *v, double *o, double *lse,
               long BH, long N, long d, int causal, double scale, int nthreads) {
    if (BH < 0 || N < 0 || d < 1) return -2;
    job_t base;
    memset(&base, 0, sizeof(base));
    base.q = q; base.k = k; base.v = v; base.o = o; base.lse = lse;
    base.BH = BH; base.N = N; base.d = d; base.causal = causal; base.scale = scale;
    base.row_begin = 0;
    job_t *jobs = (job_t *)malloc(sizeof(job_t) * (size_t)(nthreads > 0 ? nthreads : 1));
    if (!jobs) return -1;
    int rc = run_threads(&base, BH * N, nthreads, fwd_worker, jobs);
    free(jobs);
    return rc;
}

/* Decode: Nq query rows per head, each attending to all Nk keys of its head.
 * q, o: [BH][Nq][d]; k, v: [BH][Nk][d]; lse: [BH][Nq].  Returns 0 on success. */
int oracle_decode(const double *q, const double *k, const double *v, double *o, double *lse,
                  long BH, long Nq, long Nk, long d, double scale, int nthreads) {
    if (BH < 0 || Nq < 0 || Nk < 1 || d < 1) return -2;
    job_t base;
    memset(&base, 0, sizeof(base));
    base.q = q; base.k = k; base.v = v; base.o = o; base.lse = lse;
    base.BH = BH; base.N = Nk; base.Nq = Nq; base.d = d; base.scale = scale;
    base.row_begin = 0;
    job_t *jobs = (job_t *)malloc(sizeof(job_t) * (size_t)(nthreads > 0 ? nthreads : 1));
    if (!jobs) return -1;
    int rc = run_threads(&base, BH * Nq, nthreads, dec_worker, jobs);
    free(jobs);
    return rc;
}

/* Forward on selected rows only (the same rows in every head).
 * o: [BH][nrows][d], lse: [BH][nrows]. */
int oracle_fwd_rows(const double *q, const double *k, const double *v, const long *rows,
                    long nrows, double *o, double *lse, long BH, long N, long d, int causal,
                    double scale, int nthreads) {
    if (BH < 0 || N < 0 || d < 1 || nrows < 0) return -2;
    for (long r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= N) return -2;
    job_t base;
    memset(&base, 0, sizeof(base));
    base.q = q; base.k = k; base.v = v; base.o = o; base.lse = lse;
    base.BH = BH; base.N = N; base.d = d; base.causal = causal; base.scale = scale;
    base.rows = rows; base.nrows = nrows;
    base.row_begin = 0;
    job_t *jobs = (job_t *)malloc(sizeof(job_t) * (size_t)(nthreads > 0 ? nthreads : 1));
    if (!jobs) return -1;
    int rc = run_threads(&base, BH * nrows, nthreads, fwd_worker, jobs);
    free(jobs);
    return rc;
}

/* Backward of query rows [row_begin, row_end) of head bh (or of rows[row_begin ..
 * row_end) when a row list is given); dK, dV go to this thread's partial buffers,
 * dQ rows are owned by the thread and written directly (row t of the list goes to
 * dq row t in row-list mode). */
static void *bwd_worker(void *arg) {
    job_t *jb = (job_t *)arg;
    long N = jb->N, d = jb->d;
    size_t head = (size_t)jb->bh * (size_t)N * (size_t)d;
    const double *Q = jb->q + head, *K = jb->k + head, *V = jb->v + head;
    const double *dO = jb->dout + head;
    double *dQ = jb->rows ? jb->dq + (size_t)jb->bh * (size_t)jb->nrows * (size_t)d
                          : jb->dq + head;
    double *s = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    double *dp = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    memset(jb->dk_part, 0, sizeof(double) * (size_t)N * (size_t)d);
    memset(jb->dv_part, 0, sizeof(double) * (size_t)N * (size_t)d);
    for (long t = jb->row_begin; t < jb->row_end; ++t) {
        long i = jb->rows ? jb->rows[t] : t;
        long n = n_allowed(i, N, jb->causal);
        double l;
        score_row(Q + i * d, K, n, d, jb->scale, s, &l);
        const double *doi = dO + i * d;
        double Di = 0.0;
        for (long j = 0; j < n; ++j) {
            s[j] = s[j] / l; /* P_ij */
            const double *vj = V + j * d;
            double acc = 0.0;
            for (long c = 0; c < d; ++c) acc += doi[c] * vj[c];
            dp[j] = acc;     /* dP_ij */
            Di += s[j] * dp[j];
        }
        double *dqi = dQ + t * d;
        for (long c = 0; c < d; ++c) dqi[c] = 0.0;
        const double *qi = Q + i * d;
        for (long j = 0; j < n; ++j) {
            double ds = s[j] * (dp[j] - Di);       /* dS_ij */
            const double *kj = K + j * d;
            double *dkj = jb->dk_part + j * d;
            double *dvj = jb->dv_part + j * d;
            for (long c = 0; c < d; ++c) {
                dqi[c] += jb->scale * ds * kj[c];
                dkj[c] += jb->scale * ds * qi[c];
                dvj[c] += s[j] * doi[c];
            }
        }
    }
    free(s);
    free(dp);
    return NULL;
}

/* Backward over the query rows `rows` (NULL: every row) of every head.
 * dq: [BH][nrows][d] (or [BH][N][d]); dk, dv: [BH][N][d], the contributions of
 * the selected rows only. */
static int bwd_impl(const double *q, const double *k, const double *v, const double *dout,
                    const long *rows, long nrows, double *dq, double *dk, double *dv, long BH,
                    long N, long d, int causal, double scale, int nthreads) {
    if (BH < 0 || N < 0 || d < 1 || nrows < 0) return -2;
    for (long r = 0; rows && r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= N) return -2;
    long nwork = rows ? nrows : N;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > nwork) nthreads = (int)(nwork > 0 ? nwork : 1);
    size_t hsz = (size_t)N * (size_t)d;
    double *parts = (double *)malloc(sizeof(double) * hsz * 2 * (size_t)nthreads + 1);
    job_t *jobs = (job_t *)malloc(sizeof(job_t) * (size_t)nthreads);
    if (!parts || !jobs) { free(parts); free(jobs); return -1; }
    int rc = 0;
    for (long bh = 0; bh < BH && rc == 0; ++bh) {
        job_t base;
        memset(&base, 0, sizeof(base));
        base.q = q; base.k = k; base.v = v; base.dout = dout; base.dq = dq;
        base.BH = BH; base.N = N; base.d = d; base.causal = causal; base.scale = scale;
        base.bh = bh;
        base.rows = rows; base.nrows = nrows;
        pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
        if (!th) { rc = -1; break; }
        int started = 0;
        for (int t = 0; t < nthreads; ++t) {
            jobs[t] = base;
            jobs[t].row_begin = nwork * t / nthreads;
            jobs[t].row_end = nwork * (t + 1) / nthreads;
            jobs[t].dk_part = parts + hsz * (size_t)(2 * t);
            jobs[t].dv_part = parts + hsz * (size_t)(2 * t + 1);
            if (pthread_create(&th[t], NULL, bwd_worker, &jobs[t]) != 0) { rc = -1; break; }
            ++started;
        }
        for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
        free(th);
        if (rc != 0) break;
        double *dkh = dk + (size_t)bh * hsz, *dvh = dv + (size_t)bh * hsz;
        for (size_t e = 0; e < hsz; ++e) {
            double a = 0.0, b = 0.0;
            for (int t = 0; t < nthreads; ++t) {
                a += jobs[t].dk_part[e];
                b += jobs[t].dv_part[e];
            }
            dkh[e] = a;
            dvh[e] = b;
        }
    }
    free(parts);
    free(jobs);
    return rc;
}

/* Backward over every row.  dq, dk, dv: [BH][N][d]. */
int oracle_bwd(const double *q, const double *k, const double *v, const double *dout,
               double *dq, double *dk, double *dv, long BH, long N, long d, int causal,
               double scale, int nthreads) {
    return bwd_impl(q, k, v, dout, NULL, 0, dq, dk, dv, BH, N, d, causal, scale, nthreads);
}

/* Backward restricted to the query rows `rows` (the same rows in every head):
 * dq: [BH][nrows][d]; dk, dv: [BH][N][d] hold those rows' contributions. */
int oracle_bwd_rows(const double *q, const double *k, const double *v, const double *dout,
                    const long *rows, long nrows, double *dq, double *dk, double *dv, long BH,
                    long N, long d, int causal, double scale, int nthreads) {
    return bwd_impl(q, k, v, dout, rows, nrows, dq, dk, dv, BH, N, d, causal, scale, nthreads);
}
