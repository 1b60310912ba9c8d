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
 *  [L7] section 1 also lists the operators a scan accepts besides addition:
 *        multiplication, min, max, bitwise and/or, and a user-defined
 *        (maximum, number of occurrences) compound operator; [PMPP] 9.1's
 *        identity table gives 1 for multiplication, -infinity for max and
 *        +infinity for min.
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
 *    ([PMPP] 4.2 marks input[i] > threshold; [L7] section 2 keeps x > 0);
 *  - integer products, and, or, xor and the 64-bit sums are taken on the
 *    unsigned bits (wraparound modulo 2^32 or 2^64, identical bits for the
 *    signed types); xor (identity 0) is added to the listed and/or;
 *  - the infinities of the identity table are the extreme values of the
 *    integer type (max: its minimum, min: its maximum), and -inf / +inf for
 *    floats; float max and min propagate NaN (once a NaN has been seen the
 *    running value is NaN, as numpy's maximum/minimum do; this keeps -inf and
 *    +inf two-sided identities) and keep the earlier of two equal values (so
 *    -0.0 and +0.0 stay as they came);
 *  - float64 sums are accumulated with a running compensation term
 *    (Neumaier's variant of Kahan summation), so the oracle is more accurate
 *    than any fp64 scan it checks;
 *  - the (maximum, count) element is the pair (v, c) of an int32 value and a
 *    uint32 count; (v1,c1) (+) (v2,c2) is the pair with the larger value, the
 *    counts added when the values are equal; identity (INT32_MIN, 0).
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

/* ---- more operators and element types ([L7] s.1 operator list; [PMPP] 9.1
 *      identity table).  One left-to-right loop each, as above. ---- */

static uint32_t prod_u32(uint32_t acc, uint32_t x) { return acc * x; }
static uint32_t and_u32(uint32_t acc, uint32_t x) { return acc & x; }
static uint32_t or_u32(uint32_t acc, uint32_t x) { return acc | x; }
static uint32_t xor_u32(uint32_t acc, uint32_t x) { return acc ^ x; }
static int32_t min_i32(int32_t acc, int32_t x) { return x < acc ? x : acc; }
static uint32_t max_u32(uint32_t acc, uint32_t x) { return x > acc ? x : acc; }
static uint32_t min_u32(uint32_t acc, uint32_t x) { return x < acc ? x : acc; }

static uint64_t sum_u64(uint64_t acc, uint64_t x) { return acc + x; }
static uint64_t prod_u64(uint64_t acc, uint64_t x) { return acc * x; }
static uint64_t and_u64(uint64_t acc, uint64_t x) { return acc & x; }
static uint64_t or_u64(uint64_t acc, uint64_t x) { return acc | x; }
static uint64_t xor_u64(uint64_t acc, uint64_t x) { return acc ^ x; }
static int64_t max_i64(int64_t acc, int64_t x) { return x > acc ? x : acc; }
static int64_t min_i64(int64_t acc, int64_t x) { return x < acc ? x : acc; }
static uint64_t max_u64(uint64_t acc, uint64_t x) { return x > acc ? x : acc; }
static uint64_t min_u64(uint64_t acc, uint64_t x) { return x < acc ? x : acc; }

/* A NaN operand gives NaN (the earlier NaN if both are); of two equal values
 * the earlier (acc) is kept. */
static float max_f32(float acc, float x) { if (isnan(acc)) return acc; if (isnan(x)) return x; return x > acc ? x : acc; }
static float min_f32(float acc, float x) { if (isnan(acc)) return acc; if (isnan(x)) return x; return x < acc ? x : acc; }
static double max_f64(double acc, double x) { if (isnan(acc)) return acc; if (isnan(x)) return x; return x > acc ? x : acc; }
static double min_f64(double acc, double x) { if (isnan(acc)) return acc; if (isnan(x)) return x; return x < acc ? x : acc; }

/* The loop of every scan above, for one (name, type, identity, operator). */
#define ORACLE_SCAN(NAME, T, IDENT, OP)                                    \
    void oracle_scan_##NAME(const T *x, T *y, int64_t n, int exclusive)    \
    {                                                                      \
        T acc = (IDENT);                                                   \
        for (int64_t i = 0; i < n; ++i) {                                  \
            if (exclusive) {                                               \
                y[i] = acc;                                                \
                acc = OP(acc, x[i]);                                       \
            } else {                                                       \
                acc = OP(acc, x[i]);                                       \
                y[i] = acc;                                                \
            }                                                              \
        }                                                                  \
    }

ORACLE_SCAN(prod_u32, uint32_t, 1u, prod_u32)
ORACLE_SCAN(and_u32, uint32_t, 0xFFFFFFFFu, and_u32)
ORACLE_SCAN(or_u32, uint32_t, 0u, or_u32)
ORACLE_SCAN(xor_u32, uint32_t, 0u, xor_u32)
ORACLE_SCAN(min_i32, int32_t, INT32_MAX, min_i32)
ORACLE_SCAN(max_u32, uint32_t, 0u, max_u32)
ORACLE_SCAN(min_u32, uint32_t, 0xFFFFFFFFu, min_u32)
ORACLE_SCAN(sum_u64, uint64_t, 0u, sum_u64)
ORACLE_SCAN(prod_u64, uint64_t, 1u, prod_u64)
ORACLE_SCAN(and_u64, uint64_t, 0xFFFFFFFFFFFFFFFFull, and_u64)
ORACLE_SCAN(or_u64, uint64_t, 0u, or_u64)
ORACLE_SCAN(xor_u64, uint64_t, 0u, xor_u64)
ORACLE_SCAN(max_i64, int64_t, INT64_MIN, max_i64)
ORACLE_SCAN(min_i64, int64_t, INT64_MAX, min_i64)
ORACLE_SCAN(max_u64, uint64_t, 0u, max_u64)
ORACLE_SCAN(min_u64, uint64_t, 0xFFFFFFFFFFFFFFFFull, min_u64)
ORACLE_SCAN(max_f32, float, -INFINITY, max_f32)
ORACLE_SCAN(min_f32, float, INFINITY, min_f32)
ORACLE_SCAN(max_f64, double, -INFINITY, max_f64)
ORACLE_SCAN(min_f64, double, INFINITY, min_f64)

/* float64 sum: the running sum s and a compensation c holding the low-order
 * part that s lost; the prefix reported is s + c. */
void oracle_scan_sum_f64(const double *x, double *y, int64_t n, int exclusive)
{
    double s = 0.0, c = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        if (exclusive)
            y[i] = s + c;
        const double t = s + x[i];
        if (fabs(s) >= fabs(x[i]))
            c += (s - t) + x[i];
        else
            c += (x[i] - t) + s;
        s = t;
        if (!exclusive)
            y[i] = s + c;
    }
}

/* (maximum, count): x and y hold n interleaved pairs, x[2i] = value (int32
 * bits), x[2i+1] = count. */
static void maxcount(int32_t *acc_v, uint32_t *acc_c, int32_t v, uint32_t c)
{
    if (v > *acc_v) {
        *acc_v = v;
        *acc_c = c;
    } else if (v == *acc_v) {
        *acc_c = *acc_c + c;
    }
}

void oracle_scan_maxcount_i32(const uint32_t *x, uint32_t *y, int64_t n, int exclusive)
{
    int32_t acc_v = INT32_MIN;
    uint32_t acc_c = 0u;
    for (int64_t i = 0; i < n; ++i) {
        if (exclusive) {
            y[2 * i] = (uint32_t)acc_v;
            y[2 * i + 1] = acc_c;
            maxcount(&acc_v, &acc_c, (int32_t)x[2 * i], x[2 * i + 1]);
        } else {
            maxcount(&acc_v, &acc_c, (int32_t)x[2 * i], x[2 * i + 1]);
            y[2 * i] = (uint32_t)acc_v;
            y[2 * i + 1] = acc_c;
        }
    }
}

/* the float64 tolerance's scale: s[i] = |x[0]| + ... + |x[i]| */
void oracle_abs_prefix_f64(const double *x, double *s, int64_t n)
{
    double acc = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        acc = acc + fabs(x[i]);
        s[i] = acc;
    }
}

/* ---- segmented scans: head flags h[i] != 0 start a new segment (element 0
 *      always starts one); the running value restarts from the identity at
 *      each head, so y[i] is the scan of x[s..i] (inclusive) or x[s..i-1]
 *      (exclusive, the identity at s), s the last head at or before i.
 *      ([L7] section 2: each digit pass of a radix sort places its elements
 *      with a segmented scan; section 1: max/min scans answer "is this the
 *      first element of its segment that satisfies the condition") ---- */

#define ORACLE_SEGSCAN(NAME, T, IDENT, OP)                                               \
    void oracle_segscan_##NAME(const T *x, const uint8_t *h, T *y, int64_t n, int exclusive) \
    {                                                                                    \
        T acc = (IDENT);                                                                 \
        for (int64_t i = 0; i < n; ++i) {                                                \
            if (h[i])                                                                    \
                acc = (IDENT);                                                           \
            if (exclusive) {                                                             \
                y[i] = acc;                                                              \
                acc = OP(acc, x[i]);                                                     \
            } else {                                                                     \
                acc = OP(acc, x[i]);                                                     \
                y[i] = acc;                                                              \
            }                                                                            \
        }                                                                                \
    }

ORACLE_SEGSCAN(sum_u32, uint32_t, 0u, sum_u32)
ORACLE_SEGSCAN(max_i32, int32_t, INT32_MIN, max_i32)
ORACLE_SEGSCAN(prod_u32, uint32_t, 1u, prod_u32)
ORACLE_SEGSCAN(and_u32, uint32_t, 0xFFFFFFFFu, and_u32)
ORACLE_SEGSCAN(or_u32, uint32_t, 0u, or_u32)
ORACLE_SEGSCAN(xor_u32, uint32_t, 0u, xor_u32)
ORACLE_SEGSCAN(min_i32, int32_t, INT32_MAX, min_i32)
ORACLE_SEGSCAN(max_u32, uint32_t, 0u, max_u32)
ORACLE_SEGSCAN(min_u32, uint32_t, 0xFFFFFFFFu, min_u32)
ORACLE_SEGSCAN(sum_u64, uint64_t, 0u, sum_u64)
ORACLE_SEGSCAN(prod_u64, uint64_t, 1u, prod_u64)
ORACLE_SEGSCAN(and_u64, uint64_t, 0xFFFFFFFFFFFFFFFFull, and_u64)
ORACLE_SEGSCAN(or_u64, uint64_t, 0u, or_u64)
ORACLE_SEGSCAN(xor_u64, uint64_t, 0u, xor_u64)
ORACLE_SEGSCAN(max_i64, int64_t, INT64_MIN, max_i64)
ORACLE_SEGSCAN(min_i64, int64_t, INT64_MAX, min_i64)
ORACLE_SEGSCAN(max_u64, uint64_t, 0u, max_u64)
ORACLE_SEGSCAN(min_u64, uint64_t, 0xFFFFFFFFFFFFFFFFull, min_u64)
ORACLE_SEGSCAN(max_f32, float, -INFINITY, max_f32)
ORACLE_SEGSCAN(min_f32, float, INFINITY, min_f32)
ORACLE_SEGSCAN(max_f64, double, -INFINITY, max_f64)
ORACLE_SEGSCAN(min_f64, double, INFINITY, min_f64)

/* float32 sum: accumulated in fp64, as oracle_scan_sum_f32 */
void oracle_segscan_sum_f32(const float *x, const uint8_t *h, double *y, int64_t n, int exclusive)
{
    double acc = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        if (h[i])
            acc = 0.0;
        if (exclusive) {
            y[i] = acc;
            acc = acc + (double)x[i];
        } else {
            acc = acc + (double)x[i];
            y[i] = acc;
        }
    }
}

/* float64 sum: compensated, as oracle_scan_sum_f64 */
void oracle_segscan_sum_f64(const double *x, const uint8_t *h, double *y, int64_t n, int exclusive)
{
    double s = 0.0, c = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        if (h[i]) {
            s = 0.0;
            c = 0.0;
        }
        if (exclusive)
            y[i] = s + c;
        const double t = s + x[i];
        if (fabs(s) >= fabs(x[i]))
            c += (s - t) + x[i];
        else
            c += (x[i] - t) + s;
        s = t;
        if (!exclusive)
            y[i] = s + c;
    }
}

/* pairs: affine maps and (max, count), interleaved as in the plain scans */
void oracle_segscan_affine_u32(const uint32_t *x, const uint8_t *h, uint32_t *y, int64_t n, int exclusive)
{
    uint32_t acc_a = 1u, acc_b = 0u;
    for (int64_t i = 0; i < n; ++i) {
        if (h[i]) {
            acc_a = 1u;
            acc_b = 0u;
        }
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

void oracle_segscan_maxcount_i32(const uint32_t *x, const uint8_t *h, uint32_t *y, int64_t n, int exclusive)
{
    int32_t acc_v = INT32_MIN;
    uint32_t acc_c = 0u;
    for (int64_t i = 0; i < n; ++i) {
        if (h[i]) {
            acc_v = INT32_MIN;
            acc_c = 0u;
        }
        if (exclusive) {
            y[2 * i] = (uint32_t)acc_v;
            y[2 * i + 1] = acc_c;
            maxcount(&acc_v, &acc_c, (int32_t)x[2 * i], x[2 * i + 1]);
        } else {
            maxcount(&acc_v, &acc_c, (int32_t)x[2 * i], x[2 * i + 1]);
            y[2 * i] = (uint32_t)acc_v;
            y[2 * i + 1] = acc_c;
        }
    }
}

/* ---- histogram and bin offsets ([PMPP] section 4.2 lists, among the uses of
 *      scan: a radix sort's digit pass scans the digit histogram to find where
 *      each bucket starts, and converting a sparse matrix from COO to CSR scans
 *      the per-row entry counts to get the row offsets).
 *      counts[b] = number of i with bins[i] == b, for 0 <= b < nbins; entries
 *      outside [0, nbins) are not counted (the return value says how many).
 *      offsets[b] = counts[0] + ... + counts[b-1] (exclusive scan), with
 *      offsets[nbins] = the number of counted entries. ---- */

int64_t oracle_histogram(const int32_t *bins, int64_t n, int64_t nbins, int64_t *counts)
{
    int64_t outside = 0;
    for (int64_t b = 0; b < nbins; ++b)
        counts[b] = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (bins[i] >= 0 && bins[i] < nbins)
            counts[bins[i]] += 1;
        else
            outside += 1;
    }
    return outside;
}

int64_t oracle_bin_offsets(const int32_t *bins, int64_t n, int64_t nbins, int64_t *counts, int64_t *offsets)
{
    const int64_t outside = oracle_histogram(bins, n, nbins, counts);
    int64_t acc = 0;
    for (int64_t b = 0; b < nbins; ++b) {
        offsets[b] = acc;
        acc += counts[b];
    }
    offsets[nbins] = acc;
    return outside;
}

/* ---- radix sort ([L7] section 2: a radix sort makes one pass per digit, a
 *      split by the digit whose placement is a scan; [PMPP] section 4.2: the
 *      scan of the digit histogram gives where each bucket starts).  One pass:
 *      a stable counting sort of the keys by d(k) = (k >> shift) & (2^bits - 1):
 *      count each digit, exclusive-scan the counts into bucket starts, then
 *      place the keys in input order, each at the next free slot of its bucket.
 *      A full sort of 32-bit keys is four 8-bit passes, least significant first. ---- */

void oracle_radix_pass_u32(const uint32_t *in, uint32_t *out, int64_t n, int shift, int bits)
{
    const uint32_t mask = (bits >= 32) ? 0xFFFFFFFFu : ((1u << bits) - 1u);
    const int64_t nb = (int64_t)1 << bits;
    int64_t count[256] = {0};
    int64_t start[256];
    for (int64_t i = 0; i < n; ++i)
        count[(in[i] >> shift) & mask] += 1;
    int64_t acc = 0;
    for (int64_t d = 0; d < nb; ++d) {
        start[d] = acc;
        acc += count[d];
    }
    for (int64_t i = 0; i < n; ++i) {
        const uint32_t d = (in[i] >> shift) & mask;
        out[start[d]] = in[i];
        start[d] += 1;
    }
}

/* keys sorted ascending; tmp has room for n keys */
void oracle_radix_sort_u32(const uint32_t *in, uint32_t *out, uint32_t *tmp, int64_t n)
{
    oracle_radix_pass_u32(in, tmp, n, 0, 8);
    oracle_radix_pass_u32(tmp, out, n, 8, 8);
    oracle_radix_pass_u32(out, tmp, n, 16, 8);
    oracle_radix_pass_u32(tmp, out, n, 24, 8);
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
