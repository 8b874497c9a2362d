/*
 * attn_oracle.c -- plain, slow, fp64 CPU oracle for exact softmax attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only tests/, the smoke check and bench.py's CPU-baseline
 * leg use it.  It shares no code, header, table or helper with the CUDA
 * library.
 *
 * What it computes.  The lexicon page "FlashAttention" (urworte.de),
 * section "Methodische Grundlagen", paragraph "Exaktheit", states that the
 * tiled method returns the same result as the conventional computation up
 * to ordinary rounding; the glossary page "FlashAttention" (blog.brdg.mn),
 * opening paragraph, says it computes exactly what the usual implementation
 * computes.  So the oracle is that usual, materialising computation written
 * out (the "standard attention" of the page "FlashAttention-2 (DE)",
 * section "Hintergrund"), per head and per query row i:
 *
 *   z_ij  = s * sum_c q_ic k_jc                 for j in V(i)
 *   M_i   = max_j z_ij,   Z_i = sum_j exp(z_ij - M_i)
 *   P_ij  = exp(z_ij - M_i) / Z_i               (0 for j not in V(i))
 *   O_i   = sum_j P_ij v_j,   LSE_i = M_i + ln Z_i
 *
 * and the gradients of L = sum(dO * O) through that definition (softmax
 * Jacobian, no shortcut through the stored output):
 *
 *   dV_j  = sum_i P_ij dO_i
 *   dP_ij = dO_i . v_j
 *   dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik)
 *   dQ_i  = s sum_j dS_ij k_j,   dK_j = s sum_i dS_ij q_i
 *
 * V(i) is every key when causal == 0 and {j : j <= i} when causal == 1
 * (square, top-left aligned mask).  The pages write no formula; the scale s,
 * the natural-log logsumexp of the scaled scores and the mask convention are
 * the readings stated in the design notes.
 *
 * Softmax is the textbook two-pass form (max, then exponentials, then the
 * sum): it is deliberately NOT the online/running form the GPU path uses.
 *
 * Layout: every tensor is [BH][rows][d] row-major fp64; lse is [BH][Nq].
 * Work is spread over threads by (head, block of query rows).  The backward
 * pass accumulates dK/dV per row block into private buffers that are summed
 * in a fixed order afterwards, so results do not depend on thread timing.
 *
 * Return value: 0 on success, -1 on invalid arguments, -2 when memory for
 * the backward partial sums cannot be allocated.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const double *q, *k, *v, *dout;
    double *o, *lse, *dq, *dk_part, *dv_part;
    long BH, Nq, Nk, d;
    int causal;
    double scale;
    long rows_per_item; /* query rows per work item */
    long items_per_head;
    long next_item;     /* shared work counter */
    pthread_mutex_t mu;
} job_t;

static long visible_end(const job_t *J, long i)
{
    /* one past the last key row i may attend to */
    if (J->causal) {
        long e = i + 1;
        return e < J->Nk ? e : J->Nk;
    }
    return J->Nk;
}

/* Scores, max-subtracted exponentials and their sum for one query row.
 * Writes P_ij (normalised) for j < end into p and returns M_i and Z_i. */
static void softmax_row(const job_t *J, const double *qi, const double *kh,
                        long end, double *p, double *M_out, double *Z_out)
{
    long d = J->d;
    double M = -INFINITY;
    for (long j = 0; j < end; ++j) {
        double acc = 0.0;
        const double *kj = kh + j * d;
        for (long c = 0; c < d; ++c) acc += qi[c] * kj[c];
        p[j] = J->scale * acc;          /* z_ij for now */
        if (p[j] > M) M = p[j];
    }
    double Z = 0.0;
    for (long j = 0; j < end; ++j) {
        p[j] = exp(p[j] - M);
        Z += p[j];
    }
    for (long j = 0; j < end; ++j) p[j] /= Z;
    *M_out = M;
    *Z_out = Z;
}

static int take_item(job_t *J, long *item)
{
    pthread_mutex_lock(&J->mu);
    long it = J->next_item++;
    pthread_mutex_unlock(&J->mu);
    if (it >= J->BH * J->items_per_head) return 0;
    *item = it;
    return 1;
}

static void *fwd_worker(void *arg)
{
    job_t *J = (job_t *)arg;
    long d = J->d;
    double *p = (double *)malloc(sizeof(double) * (size_t)J->Nk);
    if (!p) return (void *)1;
    long item;
    while (take_item(J, &item)) {
        long h = item / J->items_per_head;
        long r0 = (item % J->items_per_head) * J->rows_per_item;
        long r1 = r0 + J->rows_per_item;
        if (r1 > J->Nq) r1 = J->Nq;
        const double *kh = J->k + h * J->Nk * d;
        const double *vh = J->v + h * J->Nk * d;
        for (long i = r0; i < r1; ++i) {
            const double *qi = J->q + (h * J->Nq + i) * d;
            double *oi = J->o + (h * J->Nq + i) * d;
            long end = visible_end(J, i);
            double M, Z;
            softmax_row(J, qi, kh, end, p, &M, &Z);
            for (long c = 0; c < d; ++c) oi[c] = 0.0;
            for (long j = 0; j < end; ++j) {
                const double *vj = vh + j * d;
                for (long c = 0; c < d; ++c) oi[c] += p[j] * vj[c];
            }
            if (J->lse) J->lse[h * J->Nq + i] = M + log(Z);
        }
    }
    free(p);
    return NULL;
}

static void *bwd_worker(void *arg)
{
    job_t *J = (job_t *)arg;
    long d = J->d;
    double *p = (double *)malloc(sizeof(double) * (size_t)J->Nk);
    double *dp = (double *)malloc(sizeof(double) * (size_t)J->Nk);
    if (!p || !dp) { free(p); free(dp); return (void *)1; }
    long item;
    while (take_item(J, &item)) {
        long h = item / J->items_per_head;
        long blk = item % J->items_per_head;
        long r0 = blk * J->rows_per_item;
        long r1 = r0 + J->rows_per_item;
        if (r1 > J->Nq) r1 = J->Nq;
        const double *kh = J->k + h * J->Nk * d;
        const double *vh = J->v + h * J->Nk * d;
        double *dkp = J->dk_part + (size_t)item * J->Nk * d;
        double *dvp = J->dv_part + (size_t)item * J->Nk * d;
        for (long i = r0; i < r1; ++i) {
            const double *qi = J->q + (h * J->Nq + i) * d;
            const double *doi = J->dout + (h * J->Nq + i) * d;
            double *dqi = J->dq + (h * J->Nq + i) * d;
            long end = visible_end(J, i);
            double M, Z;
            softmax_row(J, qi, kh, end, p, &M, &Z);
            /* dP_ij = dO_i . v_j and the Jacobian's row term sum_k P_ik dP_ik */
            double rowdot = 0.0;
            for (long j = 0; j < end; ++j) {
                const double *vj = vh + j * d;
                double acc = 0.0;
                for (long c = 0; c < d; ++c) acc += doi[c] * vj[c];
                dp[j] = acc;
                rowdot += p[j] * acc;
            }
            for (long c = 0; c < d; ++c) dqi[c] = 0.0;
            for (long j = 0; j < end; ++j) {
                double ds = p[j] * (dp[j] - rowdot);
                const double *kj = kh + j * d;
                double *dkj = dkp + j * d;
                double *dvj = dvp + j * d;
                for (long c = 0; c < d; ++c) {
                    dqi[c] += J->scale * ds * kj[c];
                    dkj[c] += J->scale * ds * qi[c];
                    dvj[c] += p[j] * doi[c];
                }
            }
        }
    }
    free(p);
    free(dp);
    return NULL;
}

static int run_threads(job_t *J, void *(*fn)(void *), int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    int started = 0, failed = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, fn, J) != 0) break;
        ++started;
    }
    if (started == 0) {
        void *r = fn(J);
        return r ? -2 : 0;
    }
    for (int t = 0; t < started; ++t) {
        void *r = NULL;
        pthread_join(th[t], &r);
        if (r) failed = 1;
    }
    return failed ? -2 : 0;
}

static int check_args(long BH, long Nq, long Nk, long d, int causal)
{
    if (BH < 1 || Nq < 1 || Nk < 1 || d < 1) return -1;
    if (causal != 0 && causal != 1) return -1;
    return 0;
}

static void init_job(job_t *J, long BH, long Nq, long Nk, long d, int causal,
                     double scale, int nthreads)
{
    memset(J, 0, sizeof(*J));
    J->BH = BH; J->Nq = Nq; J->Nk = Nk; J->d = d;
    J->causal = causal; J->scale = scale;
    /* enough row blocks per head to keep every thread busy */
    long want = (long)(nthreads > 0 ? nthreads : 1) * 4;
    long per_head = (want + BH - 1) / BH;
    if (per_head < 1) per_head = 1;
    if (per_head > Nq) per_head = Nq;
    J->rows_per_item = (Nq + per_head - 1) / per_head;
    J->items_per_head = (Nq + J->rows_per_item - 1) / J->rows_per_item;
    pthread_mutex_init(&J->mu, NULL);
}

/* Forward: o[BH][Nq][d], lse[BH][Nq] (lse may be NULL). */
int oracle_fwd(const double *q, const double *k, const double *v, double *o,
               double *lse, long BH, long Nq, long Nk, long d, int causal,
               double scale, int nthreads)
{
    if (check_args(BH, Nq, Nk, d, causal) || !q || !k || !v || !o) return -1;
    job_t J;
    init_job(&J, BH, Nq, Nk, d, causal, scale, nthreads);
    J.q = q; J.k = k; J.v = v; J.o = o; J.lse = lse;
    int rc = run_threads(&J, fwd_worker, nthreads);
    pthread_mutex_destroy(&J.mu);
    return rc;
}

/* Backward: dq[BH][Nq][d], dk/dv[BH][Nk][d] from dout[BH][Nq][d]. */
int oracle_bwd(const double *q, const double *k, const double *v,
               const double *dout, double *dq, double *dk, double *dv,
               long BH, long Nq, long Nk, long d, int causal, double scale,
               int nthreads)
{
    if (check_args(BH, Nq, Nk, d, causal) || !q || !k || !v || !dout || !dq ||
        !dk || !dv)
        return -1;
    job_t J;
    init_job(&J, BH, Nq, Nk, d, causal, scale, nthreads);
    size_t nitems = (size_t)(BH * J.items_per_head);
    size_t per = (size_t)Nk * (size_t)d;
    J.dk_part = (double *)calloc(nitems * per, sizeof(double));
    J.dv_part = (double *)calloc(nitems * per, sizeof(double));
    if (!J.dk_part || !J.dv_part) {
        free(J.dk_part); free(J.dv_part);
        pthread_mutex_destroy(&J.mu);
        return -2;
    }
    J.q = q; J.k = k; J.v = v; J.dout = dout; J.dq = dq;
    int rc = run_threads(&J, bwd_worker, nthreads);
    if (rc == 0) {
        /* fixed-order sum of the per-block partials */
        for (long h = 0; h < BH; ++h) {
            double *dkh = dk + (size_t)h * per;
            double *dvh = dv + (size_t)h * per;
            memset(dkh, 0, per * sizeof(double));
            memset(dvh, 0, per * sizeof(double));
            for (long b = 0; b < J.items_per_head; ++b) {
                size_t item = (size_t)(h * J.items_per_head + b);
                const double *pk = J.dk_part + item * per;
                const double *pv = J.dv_part + item * per;
                for (size_t x = 0; x < per; ++x) {
                    dkh[x] += pk[x];
                    dvh[x] += pv[x];
                }
            }
        }
    }
    free(J.dk_part);
    free(J.dv_part);
    pthread_mutex_destroy(&J.mu);
    return rc;
}

/* Rounding spread of the output: spread[h][i][c] = sum_j P_ij |v_jc - O_ic|
 * with P and O as above.  It bounds how far O can move when every weight
 * P_ij is perturbed by a relative amount e: |dO_ic| <= e * spread[h][i][c]
 * (the weights still summing to one), which is what rounding the weights to
 * a short format does.  Test infrastructure for deriving tolerances. */
static void *spread_worker(void *arg)
{
    job_t *J = (job_t *)arg;
    long d = J->d;
    double *p = (double *)malloc(sizeof(double) * (size_t)J->Nk);
    double *o = (double *)malloc(sizeof(double) * (size_t)d);
    if (!p || !o) { free(p); free(o); return (void *)1; }
    long item;
    while (take_item(J, &item)) {
        long h = item / J->items_per_head;
        long r0 = (item % J->items_per_head) * J->rows_per_item;
        long r1 = r0 + J->rows_per_item;
        if (r1 > J->Nq) r1 = J->Nq;
        const double *kh = J->k + h * J->Nk * d;
        const double *vh = J->v + h * J->Nk * d;
        for (long i = r0; i < r1; ++i) {
            long end = visible_end(J, i);
            double M, Z;
            softmax_row(J, J->q + (h * J->Nq + i) * d, kh, end, p, &M, &Z);
            for (long c = 0; c < d; ++c) o[c] = 0.0;
            for (long j = 0; j < end; ++j)
                for (long c = 0; c < d; ++c) o[c] += p[j] * vh[j * d + c];
            double *si = J->o + (h * J->Nq + i) * d;   /* the spread output */
            for (long c = 0; c < d; ++c) si[c] = 0.0;
            for (long j = 0; j < end; ++j)
                for (long c = 0; c < d; ++c) si[c] += p[j] * fabs(vh[j * d + c] - o[c]);
        }
    }
    free(p);
    free(o);
    return NULL;
}

int oracle_fwd_spread(const double *q, const double *k, const double *v,
                      double *spread, long BH, long Nq, long Nk, long d,
                      int causal, double scale, int nthreads)
{
    if (check_args(BH, Nq, Nk, d, causal) || !q || !k || !v || !spread) return -1;
    job_t J;
    init_job(&J, BH, Nq, Nk, d, causal, scale, nthreads);
    J.q = q; J.k = k; J.v = v; J.o = spread;
    int rc = run_threads(&J, spread_worker, nthreads);
    pthread_mutex_destroy(&J.mu);
    return rc;
}

/* The normalised probability matrix P[Nq][Nk] of one head (zeros where the
 * mask hides a key).  For small cases only: it is O(Nq*Nk) memory. */
int oracle_probs(const double *q, const double *k, double *p, long Nq, long Nk,
                 long d, int causal, double scale)
{
    if (check_args(1, Nq, Nk, d, causal) || !q || !k || !p) return -1;
    job_t J;
    init_job(&J, 1, Nq, Nk, d, causal, scale, 1);
    for (long i = 0; i < Nq; ++i) {
        double *pi = p + i * Nk;
        long end = visible_end(&J, i);
        double M, Z;
        softmax_row(&J, q + i * d, k, end, pi, &M, &Z);
        for (long j = end; j < Nk; ++j) pi[j] = 0.0;
    }
    pthread_mutex_destroy(&J.mu);
    return 0;
}
