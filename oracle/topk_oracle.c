/*
 * CPU oracle for the exact per-row bf16 top-k.  TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline /
 * reference arm may load this file's library.  The product path (the CUDA
 * library under wide_bf16_row_gb300/) never calls it, and the two share no
 * code, header, table or helper.
 *
 * Source of the definition: TensorFold PR #713, "perf(qwen27): a drafted round
 * overlaps its cache commit with the next draft, and the drafter's attention
 * and top-k use more of the GPU".
 *   - change 3 of the PR's list: every row of bf16 draft-head logits yields its
 *     best entries in (score descending, lower token index first) order;
 *   - the "Exactness" table: each row reports its entries, a count and a
 *     non-finite mask, and the cases cover ties, both zeros, NaN, infinities
 *     and padded row strides.
 * The pages leave the NaN, zero-sign, count, mask and empty-slot conventions
 * open.  The reading taken here (and by the GPU path) is:
 *   - a NaN (any sign, any payload) is never selected;
 *   - +0 and -0 are the same score, so they tie and the lower column wins;
 *     each selected entry keeps its own original bits;
 *   - +inf and -inf are ordinary extreme scores;
 *   - bf16 subnormals keep their exact values;
 *   - count = min(k, number of non-NaN columns in the row);
 *   - mask bit 0 = the row holds a NaN, bit 1 = a +inf, bit 2 = a -inf,
 *     taken over columns [0, cols) only (padding is never looked at);
 *   - slots count..k-1 hold index -1 and value bits 0x7FC0.
 *
 * Method: the plain definition.  Every value is widened to double (exact for
 * bf16), the non-NaN columns are stable-sorted by value descending with a
 * merge sort, and the first min(k, n) are reported.  Parity is pinned by the
 * tests in tests/test_oracle_pins.py (brute force, numpy's stable argsort,
 * full-sort, prefix, hand-derived fixtures and invariants).
 *
 * Build: gcc -O2 -shared -fPIC -pthread topk_oracle.c -o libtopk_oracle.so
 * Define ORACLE_MUTANT=n to build a deliberately broken variant; the pin tests
 * use those to show that each plausible mistake is caught.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* A bf16 value is the top half of an IEEE binary32; widening it to double is
 * exact. */
static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t word = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &word, sizeof f);
    return (double)f;
}

/* Does a go before b in "score descending" order?  Equal scores return 0, so
 * the merge below keeps them in column order (the lower column first). */
static int score_before(double a, double b)
{
#if ORACLE_MUTANT == 1 /* mutant: ascending order */
    return a < b;
#else
    return a > b;
#endif
}

/* Stable bottom-up merge sort of idx[0..n) by score[idx[i]] descending. */
static void stable_sort_desc(int64_t *idx, int64_t *tmp, const double *score, int64_t n)
{
    for (int64_t width = 1; width < n; width *= 2) {
        for (int64_t lo = 0; lo < n; lo += 2 * width) {
            int64_t mid = lo + width < n ? lo + width : n;
            int64_t hi = lo + 2 * width < n ? lo + 2 * width : n;
            int64_t a = lo, b = mid, o = lo;
            while (a < mid && b < hi) {
                /* take from the right run only when it is strictly better */
#if ORACLE_MUTANT == 2 /* mutant: ties go to the higher column */
                if (!score_before(score[idx[a]], score[idx[b]]))
#else
                if (score_before(score[idx[b]], score[idx[a]]))
#endif
                    tmp[o++] = idx[b++];
                else
                    tmp[o++] = idx[a++];
            }
            while (a < mid) tmp[o++] = idx[a++];
            while (b < hi) tmp[o++] = idx[b++];
        }
        memcpy(idx, tmp, (size_t)n * sizeof *idx);
    }
}

struct row_scratch {
    int64_t *idx;
    int64_t *tmp;
    double *score;
};

/* One row: x[0..cols) -> k output slots, a count and a mask. */
static void oracle_row(const uint16_t *x, int64_t cols, int32_t k, int32_t *out_idx,
                       uint16_t *out_val, int32_t *out_count, uint32_t *out_mask,
                       struct row_scratch *s)
{
    uint32_t mask = 0;
    int64_t n = 0;
#if ORACLE_MUTANT == 5 /* mutant: the last column is never looked at */
    int64_t scan = cols - 1;
#else
    int64_t scan = cols;
#endif
    for (int64_t c = 0; c < scan; ++c) {
        double v = bf16_bits_to_double(x[c]);
#if ORACLE_MUTANT == 4 /* mutant: -0 ranks below +0 */
        if (v == 0.0 && signbit(v)) v = -1e-300;
#endif
        s->score[c] = v;
        if (isnan(v)) {
            mask |= 1u;
#if ORACLE_MUTANT == 3 /* mutant: NaN is kept and ranked as +inf */
            s->score[c] = INFINITY;
            s->idx[n++] = c;
#endif
            continue;
        }
        if (isinf(v))
#if ORACLE_MUTANT == 6 /* mutant: the two infinity bits are swapped */
            mask |= v > 0 ? 4u : 2u;
#else
            mask |= v > 0 ? 2u : 4u;
#endif
        s->idx[n++] = c;
    }
    stable_sort_desc(s->idx, s->tmp, s->score, n);
    int64_t m = n < (int64_t)k ? n : (int64_t)k;
    for (int64_t i = 0; i < m; ++i) {
        out_idx[i] = (int32_t)s->idx[i];
        out_val[i] = x[s->idx[i]];
    }
    for (int64_t i = m; i < k; ++i) {
        out_idx[i] = -1;
#if ORACLE_MUTANT == 8 /* mutant: empty slots keep value bits 0 */
        out_val[i] = 0;
#else
        out_val[i] = 0x7FC0;
#endif
    }
#if ORACLE_MUTANT == 7 /* mutant: the count ignores NaN columns */
    *out_count = (int32_t)((int64_t)k < cols ? k : cols);
#else
    *out_count = (int32_t)m;
#endif
    *out_mask = mask;
}

struct job {
    const uint16_t *logits;
    int64_t row_begin, row_end, cols, row_stride;
    int32_t k;
    int32_t *out_idx;
    uint16_t *out_val;
    int32_t *out_count;
    uint32_t *out_mask;
    int status;
};

static void *run_job(void *arg)
{
    struct job *j = (struct job *)arg;
    struct row_scratch s;
    size_t n = (size_t)(j->cols > 0 ? j->cols : 1);
    s.idx = (int64_t *)malloc(n * sizeof *s.idx);
    s.tmp = (int64_t *)malloc(n * sizeof *s.tmp);
    s.score = (double *)malloc(n * sizeof *s.score);
    if (!s.idx || !s.tmp || !s.score) {
        j->status = -2;
    } else {
        for (int64_t r = j->row_begin; r < j->row_end; ++r) {
#if ORACLE_MUTANT == 9 /* mutant: rows are read as if packed (stride ignored) */
            const uint16_t *row = j->logits + r * j->cols;
#else
            const uint16_t *row = j->logits + r * j->row_stride;
#endif
            oracle_row(row, j->cols, j->k, j->out_idx + r * j->k, j->out_val + r * j->k,
                       j->out_count + r, j->out_mask + r, &s);
        }
        j->status = 0;
    }
    free(s.idx);
    free(s.tmp);
    free(s.score);
    return NULL;
}

/*
 * Exact top-k of every row of a bf16 matrix, on the host.
 *   logits      host array of bf16 bit patterns, rows x row_stride elements;
 *               columns [cols, row_stride) are padding and are never read.
 *   k           any k >= 1 (the oracle itself has no upper limit).
 *   out_idx     rows x k int32, out_val rows x k bf16 bits,
 *   out_count   rows int32, out_mask rows uint32.
 *   nthreads    worker threads (rows are split into contiguous ranges); < 1
 *               means one.
 * Returns 0, -1 for bad arguments, -2 when scratch memory cannot be had.
 */
int oracle_topk_bf16(const uint16_t *logits, int64_t rows, int64_t cols, int64_t row_stride,
                     int32_t k, int32_t *out_idx, uint16_t *out_val, int32_t *out_count,
                     uint32_t *out_mask, int32_t nthreads)
{
    if (rows < 0 || cols < 1 || row_stride < cols || k < 1) return -1;
    if (rows == 0) return 0;
    if (!logits || !out_idx || !out_val || !out_count || !out_mask) return -1;
    if (nthreads < 1) nthreads = 1;
    if ((int64_t)nthreads > rows) nthreads = (int32_t)rows;

    struct job *jobs = (struct job *)calloc((size_t)nthreads, sizeof *jobs);
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof *tids);
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return -2;
    }
    int64_t per = rows / nthreads, extra = rows % nthreads, r0 = 0;
    for (int32_t t = 0; t < nthreads; ++t) {
        int64_t cnt = per + (t < extra ? 1 : 0);
        jobs[t] = (struct job){logits, r0, r0 + cnt, cols, row_stride, k,
                               out_idx, out_val, out_count, out_mask, -3};
        r0 += cnt;
    }
    int started = 0;
    for (int32_t t = 1; t < nthreads; ++t) {
        if (pthread_create(&tids[t], NULL, run_job, &jobs[t]) != 0) break;
        started = t;
    }
    run_job(&jobs[0]);
    for (int32_t t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
    /* any range whose thread could not be started runs here */
    for (int32_t t = started + 1; t < nthreads; ++t) run_job(&jobs[t]);

    int status = 0;
    for (int32_t t = 0; t < nthreads; ++t)
        if (jobs[t].status != 0) status = jobs[t].status;
    free(jobs);
    free(tids);
    return status;
}
