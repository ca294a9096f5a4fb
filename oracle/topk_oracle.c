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
 * The same definition is applied to fp16 and fp32 logits (the pages' method
 * is stated for bf16; the other two formats keep every convention above, and
 * their empty slots hold the format's quiet NaN, 0x7E00 and 0x7FC00000).
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

enum { ORACLE_BF16 = 0, ORACLE_F16 = 1, ORACLE_F32 = 2 };

/* A bf16 value is the top half of an IEEE binary32; widening it to double is
 * exact. */
static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t word = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &word, sizeof f);
    return (double)f;
}

/* IEEE binary16: sign, 5 exponent bits (bias 15), 10 fraction bits.  Every
 * value is an integer times a power of two, so ldexp gives it exactly. */
static double f16_bits_to_double(uint16_t bits)
{
    const int sign = bits >> 15, e = (bits >> 10) & 0x1F, m = bits & 0x3FF;
    double v;
    if (e == 0x1F)
        v = m ? NAN : INFINITY;
#if ORACLE_MUTANT == 10 /* mutant: subnormals read as if normal */
    else
        v = ldexp(1024.0 + m, e - 25);
#else
    else if (e == 0)
        v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
    else
        v = ldexp(1024.0 + m, e - 25);
#endif
    return sign ? -v : v;
}

static double f32_bits_to_double(uint32_t bits)
{
#if ORACLE_MUTANT == 11 /* mutant: only the high half of an fp32 is read */
    bits &= 0xFFFF0000u;
#endif
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static size_t elem_size(int32_t dtype) { return dtype == ORACLE_F32 ? 4 : 2; }

static double elem_value(const void *row, int32_t dtype, int64_t c)
{
    if (dtype == ORACLE_F32) return f32_bits_to_double(((const uint32_t *)row)[c]);
    if (dtype == ORACLE_F16) return f16_bits_to_double(((const uint16_t *)row)[c]);
    return bf16_bits_to_double(((const uint16_t *)row)[c]);
}

/* out[i] = the original bits of row[c] */
static void elem_copy(void *out, int64_t i, const void *row, int64_t c, int32_t dtype)
{
    if (dtype == ORACLE_F32)
        ((uint32_t *)out)[i] = ((const uint32_t *)row)[c];
    else
        ((uint16_t *)out)[i] = ((const uint16_t *)row)[c];
}

/* out[i] = the empty-slot value: the format's quiet NaN */
static void elem_empty(void *out, int64_t i, int32_t dtype)
{
#if ORACLE_MUTANT == 8 /* mutant: empty slots keep value bits 0 */
    if (dtype == ORACLE_F32)
        ((uint32_t *)out)[i] = 0;
    else
        ((uint16_t *)out)[i] = 0;
#else
    if (dtype == ORACLE_F32)
        ((uint32_t *)out)[i] = 0x7FC00000u;
    else
        ((uint16_t *)out)[i] = dtype == ORACLE_F16 ? 0x7E00 : 0x7FC0;
#endif
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
static void oracle_row(const void *x, int32_t dtype, int64_t cols, int32_t k, int32_t *out_idx,
                       void *out_val, int32_t *out_count, uint32_t *out_mask, struct row_scratch *s)
{
    uint32_t mask = 0;
    int64_t n = 0;
#if ORACLE_MUTANT == 5 /* mutant: the last column is never looked at */
    int64_t scan = cols - 1;
#else
    int64_t scan = cols;
#endif
    for (int64_t c = 0; c < scan; ++c) {
        double v = elem_value(x, dtype, c);
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
        elem_copy(out_val, i, x, s->idx[i], dtype);
    }
    for (int64_t i = m; i < k; ++i) {
        out_idx[i] = -1;
        elem_empty(out_val, i, dtype);
    }
#if ORACLE_MUTANT == 7 /* mutant: the count ignores NaN columns */
    *out_count = (int32_t)((int64_t)k < cols ? k : cols);
#else
    *out_count = (int32_t)m;
#endif
    *out_mask = mask;
}

struct job {
    const unsigned char *logits;
    int32_t dtype;
    int64_t row_begin, row_end, cols, row_stride;
    int32_t k;
    int32_t *out_idx;
    unsigned char *out_val;
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
        const size_t es = elem_size(j->dtype);
        for (int64_t r = j->row_begin; r < j->row_end; ++r) {
#if ORACLE_MUTANT == 9 /* mutant: rows are read as if packed (stride ignored) */
            const unsigned char *row = j->logits + (size_t)(r * j->cols) * es;
#else
            const unsigned char *row = j->logits + (size_t)(r * j->row_stride) * es;
#endif
            oracle_row(row, j->dtype, j->cols, j->k, j->out_idx + r * j->k,
                       j->out_val + (size_t)(r * j->k) * es, j->out_count + r, j->out_mask + r, &s);
        }
        j->status = 0;
    }
    free(s.idx);
    free(s.tmp);
    free(s.score);
    return NULL;
}

/*
 * Exact top-k of every row of a bf16, fp16 or fp32 matrix, on the host.
 *   logits      host array of bit patterns, rows x row_stride elements of
 *               dtype (0 bf16, 1 fp16, 2 fp32); columns [cols, row_stride)
 *               are padding and are never read.
 *   k           any k >= 1 (the oracle itself has no upper limit).
 *   out_idx     rows x k int32, out_val rows x k elements of dtype (bits),
 *   out_count   rows int32, out_mask rows uint32.
 *   nthreads    worker threads (rows are split into contiguous ranges); < 1
 *               means one.
 * Returns 0, -1 for bad arguments, -2 when scratch memory cannot be had.
 */
int oracle_topk(const void *logits, int32_t dtype, int64_t rows, int64_t cols, int64_t row_stride, int32_t k,
                int32_t *out_idx, void *out_val, int32_t *out_count, uint32_t *out_mask, int32_t nthreads)
{
    if (rows < 0 || cols < 1 || row_stride < cols || k < 1) return -1;
    if (dtype != ORACLE_BF16 && dtype != ORACLE_F16 && dtype != ORACLE_F32) return -1;
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
        jobs[t] = (struct job){(const unsigned char *)logits, dtype, r0, r0 + cnt, cols, row_stride, k,
                               out_idx, (unsigned char *)out_val, out_count, out_mask, -3};
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
