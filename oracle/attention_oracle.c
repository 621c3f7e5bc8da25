/*
 * attention_oracle.c -- plain float64 scaled dot-product attention (CPU).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the correctness oracle that the
 * CUDA library is checked against.  Only the test suite, the smoke check and
 * the CPU-baseline leg of the bench may build, load or call it; the product
 * path never does.  It shares no code, header or constant with the CUDA path.
 *
 * What it computes (one query row at a time, every step in float64):
 *
 *   Stage 1, scores.  s_j = scale * sum_d q_d * k_{j,d}
 *       ("第 11 章 · Attention 入门" §11.1 and §11.3 step 1;
 *        "3.3 Self-Attention机制深入理解" §3.2 and §3.3).
 *   Causal mask.  Key j is visible to query row i iff j <= i + (Tk - Tq);
 *       every other key is left out of the row, which is what a score of
 *       minus infinity does ("Attention 入门" §11.1 causal bullet;
 *       "Self-Attention机制深入理解" §10.2, the 4x4 mask example).  The
 *       offset Tk - Tq aligns the last query with the last key; for Tq == Tk
 *       it is the page's lower-triangular mask.
 *   Sliding window (optional, with the causal mask).  With window W > 0 the
 *       row also drops keys more than W - 1 positions before its own, so it
 *       sees keys i + (Tk - Tq) - W + 1 .. i + (Tk - Tq): "only the most recent
 *       W tokens" ("Attention 入门" §11.8.4, Sliding Window Attention).
 *   Stage 2, safe softmax with the row maximum subtracted
 *       ("Self-Attention机制深入理解" §7.2):
 *       m = max_j s_j,  Z = sum_j exp(s_j - m),  p_j = exp(s_j - m) / Z.
 *   Stage 3, weighted sum.  o_d = sum_j p_j * v_{j,d}
 *       ("Attention 入门" §11.3 step 3; "Self-Attention机制深入理解" §3.5).
 *   Row log-sum-exp of the scaled scores: lse = m + log(Z).
 *
 * Heads: query head hq reads key/value head hq / (Hq / Hkv), which covers
 * MHA (Hq == Hkv), GQA and MQA (Hkv == 1) ("Attention 入门" §11.8.1;
 * "Self-Attention机制深入理解" §9.3).
 *
 * Layout: q is [B, Hq, Tq, D], k and v are [B, Hkv, Tk, D], all row-major
 * float32 (bf16 inputs arrive here already rounded and widened; every bf16
 * value is exact in float32).  Outputs are float64.
 *
 * The score row is materialised one query row at a time (Tk doubles per
 * thread), never the whole Tq x Tk matrix.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

typedef struct {
    const float *q, *k, *v;
    int B, Hq, Hkv, Tq, Tk, D, causal, window;
    double scale;
    const int64_t *rows; /* NULL: every row, in [B, Hq, Tq] order */
    int64_t nrows;
    double *o, *lse;
    int64_t begin, end; /* this worker's share of the row list */
    int status;
} oracle_job;

/* One query row: the three stages above, written out literally. */
static void oracle_row(const oracle_job *job, int64_t flat, double *s,
                       double *o_out, double *lse_out)
{
    const int D = job->D, Tq = job->Tq, Tk = job->Tk;
    const int64_t i = flat % Tq;
    const int64_t bh = flat / Tq;
    const int64_t hq = bh % job->Hq;
    const int64_t b = bh / job->Hq;
    const int64_t group = job->Hq / job->Hkv;
    const int64_t hkv = hq / group;

    const float *qrow = job->q + flat * (int64_t)D;
    const float *kh = job->k + (b * job->Hkv + hkv) * (int64_t)Tk * D;
    const float *vh = job->v + (b * job->Hkv + hkv) * (int64_t)Tk * D;

    /* visible keys: j0 .. n_vis-1 */
    int64_t n_vis = Tk, j0 = 0;
    if (job->causal) {
        int64_t last = i + (int64_t)(Tk - Tq);
        n_vis = last + 1 < Tk ? last + 1 : Tk;
        if (n_vis < 0) n_vis = 0;
        if (job->window > 0) {
            int64_t first = last - (int64_t)job->window + 1;
            j0 = first > 0 ? first : 0;
        }
    }

    /* Stage 1: scaled scores of the visible keys. */
    for (int64_t j = j0; j < n_vis; ++j) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d)
            acc += (double)qrow[d] * (double)kh[j * D + d];
        s[j] = job->scale * acc;
    }

    /* Stage 2: softmax with the row maximum subtracted. */
    double m = -INFINITY;
    for (int64_t j = j0; j < n_vis; ++j)
        if (s[j] > m) m = s[j];
    double z = 0.0;
    for (int64_t j = j0; j < n_vis; ++j) {
        s[j] = exp(s[j] - m);
        z += s[j];
    }
    for (int64_t j = j0; j < n_vis; ++j) s[j] /= z;

    /* Stage 3: o = P V over the visible keys. */
    for (int d = 0; d < D; ++d) o_out[d] = 0.0;
    for (int64_t j = j0; j < n_vis; ++j) {
        const double p = s[j];
        const float *vr = vh + j * D;
        for (int d = 0; d < D; ++d) o_out[d] += p * (double)vr[d];
    }
    *lse_out = n_vis > j0 ? m + log(z) : -INFINITY;
}

static void *oracle_worker(void *arg)
{
    oracle_job *job = (oracle_job *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)(job->Tk > 0 ? job->Tk : 1));
    if (!s) {
        job->status = 3;
        return NULL;
    }
    for (int64_t r = job->begin; r < job->end; ++r) {
        int64_t flat = job->rows ? job->rows[r] : r;
        oracle_row(job, flat, s, job->o + r * (int64_t)job->D, job->lse + r);
    }
    free(s);
    job->status = 0;
    return NULL;
}

/*
 * attn_oracle_f64_window: attn_oracle_f64 with a sliding window of `window`
 * keys (0: none; needs causal != 0).
 */
int attn_oracle_f64_window(const float *q, const float *k, const float *v, int B,
                           int Hq, int Hkv, int Tq, int Tk, int D, int causal,
                           int window, double scale, const int64_t *rows,
                           int64_t nrows, double *o, double *lse, int nthreads);

/*
 * attn_oracle_f64: compute attention rows in float64.
 *   rows == NULL: all B*Hq*Tq rows; o is [B,Hq,Tq,D], lse is [B,Hq,Tq].
 *   rows != NULL: nrows flat row indices (b*Hq + hq)*Tq + i; o is [nrows,D],
 *                 lse is [nrows].
 * Returns 0 on success, 1 on invalid arguments, 2 on a bad row index,
 * 3 when out of host memory.
 */
int attn_oracle_f64(const float *q, const float *k, const float *v, int B,
                    int Hq, int Hkv, int Tq, int Tk, int D, int causal,
                    double scale, const int64_t *rows, int64_t nrows,
                    double *o, double *lse, int nthreads)
{
    return attn_oracle_f64_window(q, k, v, B, Hq, Hkv, Tq, Tk, D, causal, 0, scale,
                                  rows, nrows, o, lse, nthreads);
}

int attn_oracle_f64_window(const float *q, const float *k, const float *v, int B,
                           int Hq, int Hkv, int Tq, int Tk, int D, int causal,
                           int window, double scale, const int64_t *rows,
                           int64_t nrows, double *o, double *lse, int nthreads)
{
    if (!q || !k || !v || !o || !lse) return 1;
    if (window < 0 || (window > 0 && !causal)) return 1;
    if (B < 1 || Hq < 1 || Hkv < 1 || Tq < 1 || Tk < 1 || D < 1) return 1;
    if (Hq % Hkv != 0) return 1;
    const int64_t total = (int64_t)B * Hq * Tq;
    if (rows) {
        for (int64_t r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= total) return 2;
    } else {
        nrows = total;
    }
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > nrows) nthreads = (int)(nrows > 0 ? nrows : 1);

    oracle_job jobs[256];
    pthread_t tids[256];
    int started[256];
    for (int t = 0; t < nthreads; ++t) {
        oracle_job *j = &jobs[t];
        j->q = q; j->k = k; j->v = v;
        j->B = B; j->Hq = Hq; j->Hkv = Hkv; j->Tq = Tq; j->Tk = Tk; j->D = D;
        j->causal = causal; j->window = window; j->scale = scale;
        j->rows = rows; j->nrows = nrows; j->o = o; j->lse = lse;
        j->begin = nrows * t / nthreads;
        j->end = nrows * (t + 1) / nthreads;
        j->status = 0;
        started[t] = 0;
    }
    for (int t = 1; t < nthreads; ++t)
        started[t] = pthread_create(&tids[t], NULL, oracle_worker, &jobs[t]) == 0;
    oracle_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) {
        if (started[t]) pthread_join(tids[t], NULL);
        else oracle_worker(&jobs[t]); /* thread could not start: run inline */
    }
    for (int t = 0; t < nthreads; ++t)
        if (jobs[t].status) return jobs[t].status;
    return 0;
}
