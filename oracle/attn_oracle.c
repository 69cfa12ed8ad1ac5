/*
 * Exact self-attention forward in fp64 on the CPU: the ORACLE.
 *
 * This file is test infrastructure. Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg load it; the CUDA path never does, and the two
 * share no code, header or table.
 *
 * What it computes is the plain attention graph of "From Attention Graph to
 * FlashAttention - A Memory-Centric Compilation Approach in AICF", section 1
 * (Introduction): Scores = Q x K^T, Scores = Mask(Scores), Scores =
 * Softmax(Scores), Output = Scores x V.  Per section 3 of the same page, the
 * streaming pass that the CUDA path runs changes only how that operation is
 * executed, so its result must equal this one up to rounding.  The AttenIO abstract ("I/O Analysis is All You Need", ASPLOS 2026)
 * calls the target "exact" long-sequence self-attention for the same reason.
 *
 * Readings where the pages are silent (each one is also listed in the design
 * notes):
 *   - scores are multiplied by `scale` before the mask and the softmax;
 *   - the causal mask keeps key j for query i iff j <= i, and a masked score
 *     is -infinity (it drops out of the softmax sum);
 *   - LSE_i = ln sum_j exp(scale * q_i . k_j) over the kept keys, i.e. the
 *     natural-log normaliser of the softmax, including the scale;
 *   - Q, K, V are the bf16-rounded inputs, decoded exactly to double.
 *
 * Layout: Q, K, V are [BH, N, d] arrays of bf16 bit patterns (uint16), d
 * fastest.  Outputs are double.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bf16 -> double, exactly: a bf16 value is the top half of an IEEE float. */
static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * One query row of one (batch, head): the four steps of the attention graph.
 *   q   : [d] query row (bf16 bits)
 *   Kh  : [N, d] keys of this head, Vh : [N, d] values of this head
 *   i   : the query's position (used only by the causal mask)
 *   s   : [N] scratch for the scores; on return it holds the probabilities
 *   o   : [d] output row, *lse : log-sum-exp of the scaled, masked scores
 */
static void attend_one_row(const uint16_t *q, const uint16_t *Kh, const uint16_t *Vh,
                           int64_t N, int64_t d, int64_t i, int causal, double scale,
                           double *s, double *o, double *lse)
{
    /* Scores = Q x K^T (times the scale). */
    for (int64_t j = 0; j < N; ++j) {
        const uint16_t *kj = Kh + j * d;
        double acc = 0.0;
        for (int64_t c = 0; c < d; ++c)
            acc += bf16_bits_to_double(q[c]) * bf16_bits_to_double(kj[c]);
        s[j] = scale * acc;
    }
    /* Scores = Mask(Scores): keys after the query are removed. */
    if (causal)
        for (int64_t j = i + 1; j < N; ++j)
            s[j] = -INFINITY;
    /* Scores = Softmax(Scores), with the row maximum taken out first so that
     * exp() cannot overflow; the maximum cancels in the ratio. */
    double m = -INFINITY;
    for (int64_t j = 0; j < N; ++j)
        if (s[j] > m) m = s[j];
    double l = 0.0;
    for (int64_t j = 0; j < N; ++j) {
        s[j] = exp(s[j] - m); /* exp(-inf) = 0 for masked keys */
        l += s[j];
    }
    for (int64_t j = 0; j < N; ++j)
        s[j] /= l;
    /* Output = Scores x V. */
    for (int64_t c = 0; c < d; ++c)
        o[c] = 0.0;
    for (int64_t j = 0; j < N; ++j) {
        if (s[j] == 0.0) continue;
        const uint16_t *vj = Vh + j * d;
        for (int64_t c = 0; c < d; ++c)
            o[c] += s[j] * bf16_bits_to_double(vj[c]);
    }
    *lse = m + log(l);
}

static void attend_one_row_f64(const double *q, const double *Kh, const double *Vh,
                               int64_t N, int64_t d, int64_t i, int causal, double scale,
                               double *s, double *o, double *lse);

typedef struct {
    const uint16_t *Q, *K, *V;
    const double *Qd, *Kd, *Vd; /* double inputs instead of Q, K, V when non-NULL */
    int64_t BH, N, d, R;
    int causal;
    double scale;
    const int64_t *rows; /* [BH, R] query positions, or NULL for all rows */
    double *O;           /* [BH, R, d] */
    double *LSE;         /* [BH, R] */
    double *P;           /* [BH, R, N] probabilities, or NULL */
    int64_t first, last; /* work items [first, last) of BH*R */
    int status;
} oracle_job;

static void *oracle_worker(void *arg)
{
    oracle_job *job = (oracle_job *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)(job->N > 0 ? job->N : 1));
    if (!s) { job->status = 2; return NULL; }
    for (int64_t w = job->first; w < job->last; ++w) {
        int64_t bh = w / job->R, r = w % job->R;
        int64_t i = job->rows ? job->rows[w] : r;
        if (i < 0 || i >= job->N) { job->status = 1; break; }
        const int64_t head = bh * job->N * job->d;
        if (job->Qd)
            attend_one_row_f64(job->Qd + head + i * job->d, job->Kd + head, job->Vd + head,
                               job->N, job->d, i, job->causal, job->scale, s,
                               job->O + w * job->d, job->LSE + w);
        else
            attend_one_row(job->Q + head + i * job->d, job->K + head, job->V + head,
                           job->N, job->d, i, job->causal, job->scale, s,
                           job->O + w * job->d, job->LSE + w);
        if (job->P)
            memcpy(job->P + w * job->N, s, sizeof(double) * (size_t)job->N);
    }
    free(s);
    return NULL;
}

/*
 * Attention forward for selected query rows, fp64, threaded over rows.
 *   Q, K, V   : [BH, N, d] bf16 bit patterns
 *   rows      : [BH, R] query positions per (batch, head), or NULL meaning
 *               R == N and every row in order
 *   O, LSE, P : outputs as above (P may be NULL)
 *   nthreads  : worker threads (>= 1)
 * Returns 0, or 1 for a bad argument / row index, 2 for out of memory.
 */
/* Runs the row jobs of one call on `nthreads` threads; `proto` holds the
 * inputs and outputs, the work range is filled in here. */
static int run_row_jobs(const oracle_job *proto, int nthreads)
{
    const int64_t items = proto->BH * proto->R;
    if (items == 0)
        return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > items) nthreads = (int)items;
    oracle_job *jobs = (oracle_job *)calloc((size_t)nthreads, sizeof(oracle_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) { free(jobs); free(tids); return 2; }
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = *proto;
        jobs[t].first = items * t / nthreads;
        jobs[t].last = items * (t + 1) / nthreads;
        jobs[t].status = 0;
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tids[t], NULL, oracle_worker, &jobs[t]) != 0) break;
        started = t;
    }
    oracle_worker(&jobs[0]);
    /* Threads that failed to start: run their share here. */
    for (int t = started + 1; t < nthreads; ++t)
        oracle_worker(&jobs[t]);
    int status = jobs[0].status;
    for (int t = 1; t <= started; ++t)
        pthread_join(tids[t], NULL);
    for (int t = 1; t < nthreads; ++t)
        if (jobs[t].status) status = jobs[t].status;
    free(jobs);
    free(tids);
    return status;
}

/*
 * Attention forward for selected query rows, fp64, threaded over rows.
 *   Q, K, V   : [BH, N, d] bf16 bit patterns
 *   rows      : [BH, R] query positions per (batch, head), or NULL meaning
 *               R == N and every row in order
 *   O, LSE, P : outputs as above (P may be NULL)
 *   nthreads  : worker threads (>= 1)
 * Returns 0, or 1 for a bad argument / row index, 2 for out of memory.
 */
int oracle_attn_rows(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                     int64_t BH, int64_t N, int64_t d, int causal, double scale,
                     const int64_t *rows, int64_t R,
                     double *O, double *LSE, double *P, int nthreads)
{
    if (!Q || !K || !V || !O || !LSE || BH < 0 || N < 1 || d < 1 || R < 0)
        return 1;
    if (!rows && R != N)
        return 1;
    oracle_job j = {Q, K, V, NULL, NULL, NULL, BH, N, d, R, causal, scale, rows, O, LSE, P, 0, 0, 0};
    return run_row_jobs(&j, nthreads);
}

/* The same on double-precision inputs Q, K, V [BH, N, d]. */
int oracle_attn_rows_f64(const double *Q, const double *K, const double *V,
                         int64_t BH, int64_t N, int64_t d, int causal, double scale,
                         const int64_t *rows, int64_t R,
                         double *O, double *LSE, double *P, int nthreads)
{
    if (!Q || !K || !V || !O || !LSE || BH < 0 || N < 1 || d < 1 || R < 0)
        return 1;
    if (!rows && R != N)
        return 1;
    oracle_job j = {NULL, NULL, NULL, Q, K, V, BH, N, d, R, causal, scale, rows, O, LSE, P, 0, 0, 0};
    return run_row_jobs(&j, nthreads);
}

/* ------------------------------------------------------------------------
 * 8-bit floating-point inputs.
 *
 * The FP8 forward takes Q, K, V as E4M3 codes with one fp32 scale per tensor:
 * the value of code c of tensor X is scale_X * e4m3(c).  E4M3 is the 8-bit
 * format of the OCP 8-bit Floating Point specification (OFP8): 1 sign bit, 4
 * exponent bits with bias 7, 3 mantissa bits; exponent field 0 holds the
 * subnormals m/8 * 2^-6; the code S.1111.111 is NaN; there are no infinities
 * (the largest finite value is 1.75 * 2^8 = 448).  The oracle decodes every
 * code exactly to double, applies the scale, and runs the same attention
 * graph on the decoded values.
 * ------------------------------------------------------------------------ */
static double e4m3_to_double(uint8_t code)
{
    const int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* dst[i] = scale * e4m3(src[i]) for i < n. */
int oracle_decode_e4m3(const uint8_t *src, int64_t n, double scale, double *dst)
{
    if ((!src || !dst) && n > 0) return 1;
    for (int64_t i = 0; i < n; ++i)
        dst[i] = scale * e4m3_to_double(src[i]);
    return 0;
}

/* ------------------------------------------------------------------------
 * Forward and backward on double-precision inputs.
 *
 * The backward pass is the derivative of the same attention graph with
 * respect to Q, K and V for an upstream gradient dO of the output (the LSE is
 * a saved statistic; no gradient flows into it).  With P the softmax
 * probabilities of the scaled, masked scores and O = P V:
 *     dV = P^T dO
 *     dP = dO V^T
 *     dS_ij = P_ij (dP_ij - D_i),  D_i = sum_k P_ik dP_ik = sum_c dO_ic O_ic
 *     dQ = scale * dS K,   dK = scale * dS^T Q
 * The "IO-Aware Algorithms" page describes FlashAttention's backward as
 * recomputing these activations instead of storing them; the oracle simply
 * computes them from the definition, one query row at a time.
 * ------------------------------------------------------------------------ */

/* The attention graph of one query row on double inputs (same steps as
 * attend_one_row). */
static void attend_one_row_f64(const double *q, const double *Kh, const double *Vh,
                               int64_t N, int64_t d, int64_t i, int causal, double scale,
                               double *s, double *o, double *lse)
{
    for (int64_t j = 0; j < N; ++j) {
        const double *kj = Kh + j * d;
        double acc = 0.0;
        for (int64_t c = 0; c < d; ++c)
            acc += q[c] * kj[c];
        s[j] = scale * acc;
    }
    if (causal)
        for (int64_t j = i + 1; j < N; ++j)
            s[j] = -INFINITY;
    double m = -INFINITY;
    for (int64_t j = 0; j < N; ++j)
        if (s[j] > m) m = s[j];
    double l = 0.0;
    for (int64_t j = 0; j < N; ++j) {
        s[j] = exp(s[j] - m);
        l += s[j];
    }
    for (int64_t j = 0; j < N; ++j)
        s[j] /= l;
    for (int64_t c = 0; c < d; ++c)
        o[c] = 0.0;
    for (int64_t j = 0; j < N; ++j) {
        if (s[j] == 0.0) continue;
        const double *vj = Vh + j * d;
        for (int64_t c = 0; c < d; ++c)
            o[c] += s[j] * vj[c];
    }
    *lse = m + log(l);
}

/* Forward on double inputs: O [BH, N, d], LSE [BH, N] for every row. */
int oracle_attn_f64(const double *Q, const double *K, const double *V, int64_t BH, int64_t N, int64_t d,
                    int causal, double scale, double *O, double *LSE)
{
    if (!Q || !K || !V || !O || !LSE || BH < 0 || N < 1 || d < 1) return 1;
    double *s = (double *)malloc(sizeof(double) * (size_t)N);
    if (!s) return 2;
    for (int64_t bh = 0; bh < BH; ++bh) {
        const int64_t head = bh * N * d;
        for (int64_t i = 0; i < N; ++i)
            attend_one_row_f64(Q + head + i * d, K + head, V + head, N, d, i, causal, scale, s,
                               O + head + i * d, LSE + bh * N + i);
    }
    free(s);
    return 0;
}

typedef struct {
    const double *Q, *K, *V, *dO; /* one head, [N, d] */
    int64_t N, d, first, last;    /* query rows [first, last) */
    int causal;
    double scale;
    double *dQ;                   /* [N, d], rows [first, last) written */
    double *dK, *dV;              /* [N, d] partial sums of this worker */
    int status;
} bwd_job;

static void *bwd_worker(void *arg)
{
    bwd_job *jb = (bwd_job *)arg;
    const int64_t N = jb->N, d = jb->d;
    double *p = (double *)malloc(sizeof(double) * (size_t)N);
    double *o = (double *)malloc(sizeof(double) * (size_t)d);
    if (!p || !o) { free(p); free(o); jb->status = 2; return NULL; }
    for (int64_t i = jb->first; i < jb->last; ++i) {
        const double *qi = jb->Q + i * d, *doi = jb->dO + i * d;
        double lse;
        attend_one_row_f64(qi, jb->K, jb->V, N, d, i, jb->causal, jb->scale, p, o, &lse);
        double Di = 0.0;
        for (int64_t c = 0; c < d; ++c)
            Di += doi[c] * o[c];
        double *dqi = jb->dQ + i * d;
        for (int64_t c = 0; c < d; ++c)
            dqi[c] = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            if (p[j] == 0.0) continue;
            const double *vj = jb->V + j * d, *kj = jb->K + j * d;
            double dPij = 0.0;
            for (int64_t c = 0; c < d; ++c)
                dPij += doi[c] * vj[c];
            const double dSij = p[j] * (dPij - Di);
            double *dkj = jb->dK + j * d, *dvj = jb->dV + j * d;
            for (int64_t c = 0; c < d; ++c) {
                dqi[c] += jb->scale * dSij * kj[c];
                dkj[c] += jb->scale * dSij * qi[c];
                dvj[c] += p[j] * doi[c];
            }
        }
    }
    free(p);
    free(o);
    return NULL;
}

/* Backward on double inputs for BH independent heads: dQ, dK, dV [BH, N, d]. */
int oracle_attn_bwd_f64(const double *Q, const double *K, const double *V, const double *dO, int64_t BH,
                        int64_t N, int64_t d, int causal, double scale, double *dQ, double *dK, double *dV,
                        int nthreads)
{
    if (!Q || !K || !V || !dO || !dQ || !dK || !dV || BH < 0 || N < 1 || d < 1) return 1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > N) nthreads = (int)N;
    const size_t head_elems = (size_t)N * (size_t)d;
    double *part = (double *)calloc((size_t)nthreads * 2 * head_elems, sizeof(double));
    bwd_job *jobs = (bwd_job *)calloc((size_t)nthreads, sizeof(bwd_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!part || !jobs || !tids) { free(part); free(jobs); free(tids); return 2; }
    int status = 0;
    for (int64_t bh = 0; bh < BH && !status; ++bh) {
        const size_t off = (size_t)bh * head_elems;
        memset(part, 0, (size_t)nthreads * 2 * head_elems * sizeof(double));
        for (int t = 0; t < nthreads; ++t) {
            bwd_job jb = {Q + off, K + off, V + off, dO + off, N, d, N * t / nthreads, N * (t + 1) / nthreads,
                          causal, scale, dQ + off, part + (size_t)(2 * t) * head_elems,
                          part + (size_t)(2 * t + 1) * head_elems, 0};
            jobs[t] = jb;
        }
        int started = 0;
        for (int t = 1; t < nthreads; ++t) {
            if (pthread_create(&tids[t], NULL, bwd_worker, &jobs[t]) != 0) break;
            started = t;
        }
        bwd_worker(&jobs[0]);
        for (int t = started + 1; t < nthreads; ++t)
            bwd_worker(&jobs[t]);
        for (int t = 1; t <= started; ++t)
            pthread_join(tids[t], NULL);
        for (int t = 0; t < nthreads; ++t)
            if (jobs[t].status) status = jobs[t].status;
        for (size_t e = 0; e < head_elems; ++e) {
            double sk = 0.0, sv = 0.0;
            for (int t = 0; t < nthreads; ++t) {
                sk += part[(size_t)(2 * t) * head_elems + e];
                sv += part[(size_t)(2 * t + 1) * head_elems + e];
            }
            dK[off + e] = sk;
            dV[off + e] = sv;
        }
    }
    free(part);
    free(jobs);
    free(tids);
    return status;
}

/* ------------------------------------------------------------------------
 * Standalone row operations ("Softmax streaming" and "LayerNorm streaming" in
 * the outlook of "From Attention Graph to FlashAttention - A Memory-Centric
 * Compilation Approach in AICF", section 8).  The oracle computes each from its
 * plain definition, row by row, in fp64.
 * ------------------------------------------------------------------------ */

/* Y[r, i] = exp(X[r, i] - max_j X[r, j]) / sum_j exp(X[r, j] - max_j X[r, j]). */
int oracle_softmax_rows(const double *X, int64_t R, int64_t N, double *Y)
{
    if (!X || !Y || R < 0 || N < 1) return 1;
    for (int64_t r = 0; r < R; ++r) {
        const double *x = X + r * N;
        double *y = Y + r * N;
        double m = -INFINITY;
        for (int64_t j = 0; j < N; ++j)
            if (x[j] > m) m = x[j];
        double l = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            y[j] = exp(x[j] - m);
            l += y[j];
        }
        for (int64_t j = 0; j < N; ++j)
            y[j] /= l;
    }
    return 0;
}

/* Layer normalisation of each row:
 *   mean = sum_j x_j / N,  var = sum_j (x_j - mean)^2 / N  (the population variance),
 *   Y[r, i] = (x_i - mean) / sqrt(var + eps) * gamma[i] + beta[i]. */
int oracle_layernorm_rows(const double *X, const double *gamma, const double *beta, int64_t R, int64_t N,
                          double eps, double *Y)
{
    if (!X || !gamma || !beta || !Y || R < 0 || N < 1 || !(eps >= 0.0)) return 1;
    for (int64_t r = 0; r < R; ++r) {
        const double *x = X + r * N;
        double *y = Y + r * N;
        double mean = 0.0;
        for (int64_t j = 0; j < N; ++j)
            mean += x[j];
        mean /= (double)N;
        double var = 0.0;
        for (int64_t j = 0; j < N; ++j)
            var += (x[j] - mean) * (x[j] - mean);
        var /= (double)N;
        const double rstd = 1.0 / sqrt(var + eps);
        for (int64_t j = 0; j < N; ++j)
            y[j] = (x[j] - mean) * rstd * gamma[j] + beta[j];
    }
    return 0;
}
