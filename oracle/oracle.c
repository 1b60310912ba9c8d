/*
 * oracle.c -- sequential CPU oracle for the device-wide scan and the stream
 * compaction built on it.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the CPU-baseline leg
 * of the benchmark do. It shares no header, helper, table or constant with
 * the CUDA path.
 *
 * Every function is the plain definition written out as one left-to-right
 * loop, with no blocking, no reordering and no parallelism, so that it can be
 * checked against the pages by eye.
 *
 * Sources (page title, section):
 *  [L7]  "Lecture 7: Parallel pattern -- prefix sum / scan: double buffering
 *        and hierarchical algorithms" (UIUC ECE408 course notes, runguoli.com),
 *        section 1 "Scan: inclusive and exclusive" and section 2
 *        "Applications of Scan" (stream compaction).
 *  [TUT] "CUDA programming: parallel prefix-sum scan explained"
 *        (m.youleyou.com), sections 2.1 Inclusive Scan, 2.2 Exclusive Scan and
 *        section 3 (the serial recurrence out[i] = out[i-1] + in[i-1]).
 *  [PMPP] "Chapter 9 Parallel Patterns: Prefix Sum - Scan Algorithms"
 *        (bittern.cn), section 9.1 (definition, identity table) and section
 *        9.6 "Applications of Scan" (filtering).
 *
 * Readings where the pages leave a step open:
 *  - integer sums wrap modulo 2^32 (both int32 and uint32 are summed as
 *    uint32_t, which is exact two's complement wraparound in C);
 *  - the identity of int32 max is INT32_MIN (the table in [PMPP] 9.1 says
 *    minus infinity);
 *  - an affine element (a, b) is the map h -> a*h + b (mod 2^32); the scan
 *    applies the earlier element first, which fixes the non-commutative order
 *    that [L7] section 1 says a scan keeps;
 *  - float32 inputs are accumulated in fp64 (the CPU references in [L7]'s
 *    programs accumulate in double);
 *  - the compaction predicate is "x <op> threshold" evaluated in double
 *    ([PMPP] 4.2 marks input[i] > threshold; [L7] section 2 keeps x > 0).
 */
#include <stdint.h>
#include <math.h>

/* ---- operators and identities ([L7] s.1; [PMPP] 9.1 identity table) ---- */

static uint32_t sum_u32(uint32_t acc, uint32_t x) { return acc + x; }

static int32_t max_i32(int32_t acc, int32_t x) { return x > acc ? x : acc; }

/* (a1,b1) then (a2,b2): h -> a2*(a1*h + b1) + b2 = (a2*a1)*h + (a2*b1 + b2). */
static void compose_affine(uint32_t *acc_a, uint32_t *acc_b, uint32_t a, uint32_t b)
{
    uint32_t na = a * *acc_a;
    uint32_t nb = a * *acc_b + b;
    *acc_a = na;
    *acc_b = nb;
}

/* ---- scans: inclusive y[i] = x[0] (+) ... (+) x[i];
 *             exclusive y[0] = I, y[i] = x[0] (+) ... (+) x[i-1]
 *      ([L7] s.1; [TUT] 2.1/2.2/3; [PMPP] 9.1) ---- */

void oracle_scan_sum_u32(const uint32_t *x, uint32_t *y, int64_t n, int exclusive)
{
    uint32_t acc = 0u;
    for (int64_t i = 0; i < n; ++i) {
        if (exclusive) {
            y[i] = acc;
            acc = sum_u32(acc, x[i]);
        } else {
            acc = sum_u32(acc, x[i]);
            y[i] = acc;
        }
    }
}

void oracle_scan_sum_f32(const float *x, double *y, int64_t n, int exclusive)
{
    double acc = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        if (exclusive) {
            y[i] = acc;
            acc = acc + (double)x[i];
        } else {
            acc = acc + (double)x[i];
            y[i] = acc;
        }
    }
}

void oracle_scan_max_i32(const int32_t *x, int32_t *y, int64_t n, int exclusive)
{
    int32_t acc = INT32_MIN;
    for (int64_t i = 0; i < n; ++i) {
        if (exclusive) {
            y[i] = acc;
            acc = max_i32(acc, x[i]);
        } else {
            acc = max_i32(acc, x[i]);
            y[i] = acc;
        }
    }
}

/* x and y hold n interleaved pairs: x[2i] = a_i, x[2i+1] = b_i. */
void oracle_scan_affine_u32(const uint32_t *x, uint32_t *y, int64_t n, int exclusive)
{
    uint32_t acc_a = 1u, acc_b = 0u;
    for (int64_t i = 0; i < n; ++i) {
        if (exclusive) {
            y[2 * i] = acc_a;
            y[2 * i + 1] = acc_b;
            compose_affine(&acc_a, &acc_b, x[2 * i], x[2 * i + 1]);
        } else {
            compose_affine(&acc_a, &acc_b, x[2 * i], x[2 * i + 1]);
            y[2 * i] = acc_a;
            y[2 * i + 1] = acc_b;
        }
    }
}

/* ---- batched rows: the same scan on each row of a row-major rows x cols
 *      matrix, the accumulator starting again from the identity at each row
 *      (no passage on the pages; the plain reading of "independent scans") ---- */

void oracle_scan_batched_sum_u32(const uint32_t *x, uint32_t *y, int64_t rows, int64_t cols, int exclusive)
{
    for (int64_t r = 0; r < rows; ++r)
        oracle_scan_sum_u32(x + r * cols, y + r * cols, cols, exclusive);
}

void oracle_scan_batched_sum_f32(const float *x, double *y, int64_t rows, int64_t cols, int exclusive)
{
    for (int64_t r = 0; r < rows; ++r)
        oracle_scan_sum_f32(x + r * cols, y + r * cols, cols, exclusive);
}

void oracle_scan_batched_max_i32(const int32_t *x, int32_t *y, int64_t rows, int64_t cols, int exclusive)
{
    for (int64_t r = 0; r < rows; ++r)
        oracle_scan_max_i32(x + r * cols, y + r * cols, cols, exclusive);
}

void oracle_scan_batched_affine_u32(const uint32_t *x, uint32_t *y, int64_t rows, int64_t cols, int exclusive)
{
    for (int64_t r = 0; r < rows; ++r)
        oracle_scan_affine_u32(x + 2 * r * cols, y + 2 * r * cols, cols, exclusive);
}

/* ---- stream compaction ([L7] s.2; [PMPP] 9.6 and 4.2):
 *      keep x[i] when pred(x[i]) holds, in input order; return the count ---- */

enum { PRED_GT = 0, PRED_GE = 1, PRED_LT = 2, PRED_LE = 3, PRED_EQ = 4, PRED_NE = 5 };

static int keep(double v, int pred, double t)
{
    switch (pred) {
    case PRED_GT: return v > t;
    case PRED_GE: return v >= t;
    case PRED_LT: return v < t;
    case PRED_LE: return v <= t;
    case PRED_EQ: return v == t;
    case PRED_NE: return v != t;
    default: return 0;
    }
}

int64_t oracle_compact_i32(const int32_t *x, int64_t n, int pred, double t, int32_t *out)
{
    int64_t c = 0;
    for (int64_t i = 0; i < n; ++i)
        if (keep((double)x[i], pred, t))
            out[c++] = x[i];
    return c;
}

int64_t oracle_compact_u32(const uint32_t *x, int64_t n, int pred, double t, uint32_t *out)
{
    int64_t c = 0;
    for (int64_t i = 0; i < n; ++i)
        if (keep((double)x[i], pred, t))
            out[c++] = x[i];
    return c;
}

int64_t oracle_compact_f32(const float *x, int64_t n, int pred, double t, float *out)
{
    int64_t c = 0;
    for (int64_t i = 0; i < n; ++i)
        if (keep((double)x[i], pred, t))
            out[c++] = x[i];
    return c;
}

/* ---- the float32 tolerance's scale: s[i] = |x[0]| + ... + |x[i]| in fp64 ---- */

void oracle_abs_prefix_f32(const float *x, double *s, int64_t n)
{
    double acc = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        acc = acc + fabs((double)x[i]);
        s[i] = acc;
    }
}
