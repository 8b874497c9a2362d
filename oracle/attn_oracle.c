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

/* ------------------------------------------------------------------ FP8
 *
 * The FP8 forward.  The page "FlashAttention-2 (DE)", section
 * "Vergleich mit nachfolgenden Versionen" / "FlashAttention-3", names FP8
 * (low precision) as one of FlashAttention-3's additions and gives no
 * formula.  The reading implemented here (and by the GPU path):
 *
 *  - Q, K, V arrive as e4m3 codes q8, k8, v8 with one scale per tensor:
 *    the value of code c of tensor X is e4m3_value(c) * sX.
 *  - Scores are exact on those values: x_ij = s * log2(e) * sum_c q_ic k_jc
 *    (log2 units), x_ij = -inf for keys the mask hides.
 *  - M_i = ceil(max_j x_ij), an integer.  The weight that multiplies v_j is
 *    the probability rounded to e4m3 at that power-of-two scale:
 *    w_ij = e4m3_round(2^(x_ij - M_i + 8)), a value in [0, 256].
 *  - O_i = sv * sum_j w_ij v_j / sum_j w_ij (the rounded weights are what
 *    is applied, and they are normalised by their own sum);
 *    LSE_i = ln(2) * (M_i - 8 + log2 sum_j 2^(x_ij - M_i + 8)), the exact
 *    logsumexp of the scaled scores.
 *
 * Because M_i is an integer and e4m3 rounding commutes with multiplication
 * by a power of two while the value stays in the normal range, the weights
 * do not depend on how a tiled implementation walks the keys (the running
 * maximum it uses is an integer too).  Only weights below the normal range
 * (2^(x - M + 8) < 2^-6) do; oracle_fwd_fp8 reports a per-element bound
 * for them and for weights whose rounding the GPU's fp32 scores could tip.
 *
 * The e4m3 format: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits;
 * exponent field 0 holds the subnormals m * 2^-9; exponent 15 with mantissa
 * 7 is NaN; there are no infinities; the largest finite value is 448.
 */

double e4m3_value(unsigned char code)
{
    int sgn = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return sgn ? -v : v;
}

/* Nearest e4m3 value to x, ties to the even mantissa, magnitudes above 448
 * saturated to 448 (the GPU converts with saturation to the finite range). */
double e4m3_round(double x)
{
    if (isnan(x)) return NAN;
    double a = fabs(x);
    if (a == 0.0) return x;
    int ex;
    frexp(a, &ex);                     /* a = f * 2^ex, f in [0.5, 1) */
    int e = ex - 1;                    /* binade: 2^e <= a < 2^(e+1) */
    if (e < -6) e = -6;                /* subnormal spacing below 2^-6 */
    double ulp = ldexp(1.0, e - 3);
    double r = nearbyint(a / ulp) * ulp;   /* default rounding: ties to even */
    if (r > 448.0) r = 448.0;
    return x < 0 ? -r : r;
}

typedef struct {
    const unsigned char *q8, *k8, *v8;
    double sq, sk, sv;
    double *o, *lse, *bound;
    long BH, Nq, Nk, d;
    int causal;
    double scale;
    double acc_rel;     /* relative precision assumed for the GPU's fp32 score sums */
    int stale;          /* binades by which the GPU's running maximum may lag the row maximum */
    double *x_out, *w_out, *delta_out, *M_out;   /* optional per-key detail: [BH][Nq][Nk], M [BH][Nq] */
    long rows_per_item, items_per_head, next_item;
    pthread_mutex_t mu;
} fp8_job_t;

static int fp8_take(fp8_job_t *J, long *item)
{
    pthread_mutex_lock(&J->mu);
    long it = J->next_item++;
    pthread_mutex_unlock(&J->mu);
    if (it >= J->BH * J->items_per_head) return 0;
    *item = it;
    return 1;
}

static void *fp8_worker(void *arg)
{
    fp8_job_t *J = (fp8_job_t *)arg;
    const long d = J->d;
    const double c = J->scale * J->sq * J->sk / log(2.0);   /* s * log2(e) * sq * sk */
    double *x = (double *)malloc(sizeof(double) * (size_t)J->Nk);
    double *w = (double *)malloc(sizeof(double) * (size_t)J->Nk);
    double *dw = (double *)malloc(sizeof(double) * (size_t)J->Nk);
    double *qd = (double *)malloc(sizeof(double) * (size_t)d);
    double *vd = (double *)malloc(sizeof(double) * (size_t)J->Nk * d);
    if (!x || !w || !dw || !qd || !vd) { free(x); free(w); free(dw); free(qd); free(vd); return (void *)1; }
    long item;
    long vh_loaded = -1;
    while (fp8_take(J, &item)) {
        long h = item / J->items_per_head;
        long r0 = (item % J->items_per_head) * J->rows_per_item;
        long r1 = r0 + J->rows_per_item;
        if (r1 > J->Nq) r1 = J->Nq;
        const unsigned char *kh = J->k8 + h * J->Nk * d;
        if (vh_loaded != h) {
            const unsigned char *vh = J->v8 + h * J->Nk * d;
            for (long t = 0; t < J->Nk * d; ++t) vd[t] = e4m3_value(vh[t]);
            vh_loaded = h;
        }
        for (long i = r0; i < r1; ++i) {
            const unsigned char *qi = J->q8 + (h * J->Nq + i) * d;
            for (long cc = 0; cc < d; ++cc) qd[cc] = e4m3_value(qi[cc]);
            long end = J->causal ? (i + 1 < J->Nk ? i + 1 : J->Nk) : J->Nk;
            double mx = -INFINITY;
            for (long j = 0; j < end; ++j) {
                const unsigned char *kj = kh + j * d;
                double acc = 0.0, mag = 0.0;
                for (long cc = 0; cc < d; ++cc) {
                    double t = qd[cc] * e4m3_value(kj[cc]);
                    acc += t;
                    mag += fabs(t);
                }
                x[j] = c * acc;
                dw[j] = fabs(c) * mag;      /* for the bound below */
                if (x[j] > mx) mx = x[j];
            }
            double M = ceil(mx);
            double W = 0.0, Z = 0.0;
            for (long j = 0; j < end; ++j) {
                double y = exp2(x[j] - M + 8.0);
                w[j] = e4m3_round(y);
                W += w[j];
                Z += y;
                /* Bound on |w_gpu - w_oracle|: the GPU computes y from fp32
                 * scores (error <= acc_rel * |c| * sum|q k| + 2^-23 |x|) and
                 * exp2 in fp32 (relative 2^-21): if y lies that close to a
                 * rounding midpoint, its rounding may go the other way (one
                 * ulp).  Below the normal range (shifted up by the lag
                 * `stale` its running maximum may have, plus one binade of
                 * margin), the GPU rounds on a grid that depends on that
                 * maximum: at most one subnormal step of the GPU's scale. */
                double dx = J->acc_rel * dw[j] + ldexp(fabs(x[j]), -23);
                double rel = 0.6931471805599453 * dx + ldexp(1.0, -21);
                double delta = 0.0;
                if (y < ldexp(1.0, -5 + J->stale)) {
                    delta = ldexp(1.0, -9 + J->stale);
                } else {
                    int ex;
                    frexp(y, &ex);
                    double ulp = ldexp(1.0, ex - 1 - 3);
                    double mid = (floor(y / ulp) + 0.5) * ulp;
                    if (fabs(y - mid) <= rel * y) delta = ulp;
                }
                dw[j] = delta;
            }
            if (J->w_out) {
                const long base = (h * J->Nq + i) * J->Nk;
                for (long j = 0; j < J->Nk; ++j) {
                    const int vis = j < end;
                    J->x_out[base + j] = vis ? x[j] : -INFINITY;
                    J->w_out[base + j] = vis ? w[j] : 0.0;
                    J->delta_out[base + j] = vis ? dw[j] : 0.0;
                }
                J->M_out[h * J->Nq + i] = M;
            }
            double *oi = J->o + (h * J->Nq + i) * d;
            for (long cc = 0; cc < d; ++cc) {
                double acc = 0.0;
                for (long j = 0; j < end; ++j) acc += w[j] * vd[j * d + cc];
                oi[cc] = J->sv * acc / W;
            }
            if (J->lse) J->lse[h * J->Nq + i] = log(2.0) * (M - 8.0 + log2(Z));
            if (J->bound) {
                double dsum = 0.0;
                for (long j = 0; j < end; ++j) dsum += dw[j];
                double *bi = J->bound + (h * J->Nq + i) * d;
                for (long cc = 0; cc < d; ++cc) {
                    double o_c = oi[cc] / J->sv, b = 0.0;
                    for (long j = 0; j < end; ++j)
                        if (dw[j] > 0.0) b += dw[j] * fabs(vd[j * d + cc] - o_c);
                    bi[cc] = (W - dsum > 0.0) ? fabs(J->sv) * b / (W - dsum) : INFINITY;
                }
            }
        }
    }
    free(x); free(w); free(dw); free(qd); free(vd);
    return NULL;
}

/* FP8 forward of e4m3 codes q8[BH][Nq][d], k8/v8[BH][Nk][d] with tensor
 * scales sq, sk, sv: o[BH][Nq][d], lse[BH][Nq] (may be NULL) as defined
 * above, and optionally bound[BH][Nq][d]: how far a GPU result may lie from
 * o because of the weights whose rounding the GPU may take differently
 * (acc_rel = relative precision of the GPU's fp32 score sums; stale = how
 * many binades its running maximum may lag the row maximum). */
int oracle_fwd_fp8_detail(const unsigned char *q8, const unsigned char *k8, const unsigned char *v8,
                          double sq, double sk, double sv, double *o, double *lse, double *bound,
                          long BH, long Nq, long Nk, long d, int causal, double scale, double acc_rel,
                          int stale, int nthreads, double *x_out, double *w_out, double *delta_out,
                          double *M_out);

int oracle_fwd_fp8(const unsigned char *q8, const unsigned char *k8, const unsigned char *v8,
                   double sq, double sk, double sv, double *o, double *lse, double *bound,
                   long BH, long Nq, long Nk, long d, int causal, double scale, double acc_rel,
                   int stale, int nthreads)
{
    return oracle_fwd_fp8_detail(q8, k8, v8, sq, sk, sv, o, lse, bound, BH, Nq, Nk, d, causal, scale,
                                 acc_rel, stale, nthreads, NULL, NULL, NULL, NULL);
}

/* The same, also returning for every (row, key) the score x (log2 units,
 * -inf where masked), the rounded weight w and the change delta that the
 * bound allows for it, and each row's M: x_out, w_out, delta_out
 * [BH][Nq][Nk] and M_out [BH][Nq], all four or none.  For small tests. */
int oracle_fwd_fp8_detail(const unsigned char *q8, const unsigned char *k8, const unsigned char *v8,
                          double sq, double sk, double sv, double *o, double *lse, double *bound,
                          long BH, long Nq, long Nk, long d, int causal, double scale, double acc_rel,
                          int stale, int nthreads, double *x_out, double *w_out, double *delta_out,
                          double *M_out)
{
    if (check_args(BH, Nq, Nk, d, causal) || !q8 || !k8 || !v8 || !o) return -1;
    if ((x_out || w_out || delta_out || M_out) && !(x_out && w_out && delta_out && M_out)) return -1;
    fp8_job_t J;
    memset(&J, 0, sizeof(J));
    J.x_out = x_out; J.w_out = w_out; J.delta_out = delta_out; J.M_out = M_out;
    J.q8 = q8; J.k8 = k8; J.v8 = v8;
    J.sq = sq; J.sk = sk; J.sv = sv;
    J.o = o; J.lse = lse; J.bound = bound;
    J.BH = BH; J.Nq = Nq; J.Nk = Nk; J.d = d;
    J.causal = causal; J.scale = scale; J.acc_rel = acc_rel; J.stale = stale < 0 ? 0 : stale;
    long want = (long)(nthreads > 0 ? nthreads : 1) * 4;
    long per_head = (want + BH - 1) / BH;
    if (per_head < 1) per_head = 1;
    if (per_head > Nq) per_head = Nq;
    J.rows_per_item = (Nq + per_head - 1) / per_head;
    J.items_per_head = (Nq + J.rows_per_item - 1) / J.rows_per_item;
    pthread_mutex_init(&J.mu, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    int started = 0, failed = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, fp8_worker, &J) != 0) break;
        ++started;
    }
    if (started == 0) failed = fp8_worker(&J) != NULL;
    for (int t = 0; t < started; ++t) {
        void *r = NULL;
        pthread_join(th[t], &r);
        if (r) failed = 1;
    }
    pthread_mutex_destroy(&J.mu);
    return failed ? -2 : 0;
}
