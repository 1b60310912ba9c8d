"""Plant plausible mistakes in copies of the oracle and check that the pins catch each.

Each mutant is oracle.c with one textual change, compiled with gcc into a
temporary directory.  The real oracle source is never modified.
"""
import os

import pytest

import oracle
from oracle_pins import ALL_PINS

MUTANTS = {
    # exclusive scan writes after accumulating (i.e. emits the inclusive value)
    "exclusive_is_inclusive": ("            y[i] = acc;\n            acc = sum_u32(acc, x[i]);",
                               "            acc = sum_u32(acc, x[i]);\n            y[i] = acc;"),
    # a dropped term: the first element is skipped
    "dropped_first_term": ("    uint32_t acc = 0u;\n    for (int64_t i = 0; i < n; ++i) {",
                           "    uint32_t acc = 0u;\n    for (int64_t i = 0; i < n; ++i) { if (i == 0 && n > 3) { y[0] = exclusive ? 0u : 0u; continue; }"),
    # wrong identity for max
    "max_identity_zero": ("    int32_t acc = INT32_MIN;", "    int32_t acc = 0;"),
    # max replaced by min-like comparison
    "max_wrong_sign": ("return x > acc ? x : acc;", "return x < acc ? x : acc;"),
    # affine composition in the wrong order (later map applied first)
    "affine_order_swapped": ("    uint32_t na = a * *acc_a;\n    uint32_t nb = a * *acc_b + b;",
                             "    uint32_t na = *acc_a * a;\n    uint32_t nb = *acc_a * b + *acc_b;"),
    # affine: transposed operand in the offset term
    "affine_transposed": ("    uint32_t nb = a * *acc_b + b;", "    uint32_t nb = *acc_a * *acc_b + b;"),
    # float accumulated in float32
    "float_in_f32": ("            acc = acc + (double)x[i];\n            y[i] = acc;",
                     "            acc = (float)(acc + (double)x[i]);\n            y[i] = acc;"),
    # compaction predicate off by one (>= instead of >)
    "pred_gt_is_ge": ("    case PRED_GT: return v > t;", "    case PRED_GT: return v >= t;"),
    # batched rows: wrong row stride
    "batched_row_stride": ("        oracle_scan_sum_u32(x + r * cols, y + r * cols, cols, exclusive);",
                           "        oracle_scan_sum_u32(x + r * cols, y + r * cols, cols - (cols > 1), exclusive);"),
    # abs prefix without the absolute value
    "abs_prefix_signed": ("        acc = acc + fabs((double)x[i]);", "        acc = acc + (double)x[i];"),
    # wrong identity for int32 min
    "min_identity_zero": ("ORACLE_SCAN(min_i32, int32_t, INT32_MAX, min_i32)", "ORACLE_SCAN(min_i32, int32_t, 0, min_i32)"),
    # wrong identity for the 64-bit product
    "prod_identity_zero": ("ORACLE_SCAN(prod_u64, uint64_t, 1u, prod_u64)", "ORACLE_SCAN(prod_u64, uint64_t, 0u, prod_u64)"),
    # xor written as or
    "xor_is_or": ("static uint32_t xor_u32(uint32_t acc, uint32_t x) { return acc ^ x; }",
                  "static uint32_t xor_u32(uint32_t acc, uint32_t x) { return acc | x; }"),
    # unsigned max compared as signed
    "max_u32_signed": ("static uint32_t max_u32(uint32_t acc, uint32_t x) { return x > acc ? x : acc; }",
                       "static uint32_t max_u32(uint32_t acc, uint32_t x) { return (int32_t)x > (int32_t)acc ? x : acc; }"),
    # 64-bit sum truncated to 32 bits
    "sum_u64_truncated": ("static uint64_t sum_u64(uint64_t acc, uint64_t x) { return acc + x; }",
                          "static uint64_t sum_u64(uint64_t acc, uint64_t x) { return (uint32_t)(acc + x); }"),
    # float64 sum without its compensation term
    "f64_sum_uncompensated": ("        if (!exclusive)\n            y[i] = s + c;", "        if (!exclusive)\n            y[i] = s;"),
    # float max that ignores NaN instead of propagating it
    "fmax_ignores_nan": ("static float max_f32(float acc, float x) { if (isnan(acc)) return acc; if (isnan(x)) return x;",
                         "static float max_f32(float acc, float x) { if (isnan(acc)) return x; if (isnan(x)) return acc;"),
    # float min keeping the later of two equal values
    "fmin_tie_later": ("static double min_f64(double acc, double x) { if (isnan(acc)) return acc; if (isnan(x)) return x; return x < acc ? x : acc; }",
                       "static double min_f64(double acc, double x) { if (isnan(acc)) return acc; if (isnan(x)) return x; return x <= acc ? x : acc; }"),
    # (max, count): equal values do not add their counts
    "maxcount_ties_not_added": ("        *acc_c = *acc_c + c;", "        *acc_c = c;"),
    # bin offsets that include the bin's own count (inclusive instead of exclusive)
    "bin_offsets_inclusive": ("        offsets[b] = acc;\n        acc += counts[b];", "        acc += counts[b];\n        offsets[b] = acc;"),
    # histogram that drops bin 0
    "histogram_drops_bin0": ("        if (bins[i] >= 0 && bins[i] < nbins)", "        if (bins[i] > 0 && bins[i] < nbins)"),
    # radix pass that places keys in reverse input order inside a bucket (not stable)
    "radix_not_stable": ("        out[start[d]] = in[i];\n        start[d] += 1;",
                         "        out[start[d] + count[d] - 1] = in[i];\n        count[d] -= 1;"),
    # radix sort whose passes run most significant digit first
    "radix_msd_first": ("    oracle_radix_pass_u32(in, tmp, n, 0, 8);\n    oracle_radix_pass_u32(tmp, out, n, 8, 8);",
                        "    oracle_radix_pass_u32(in, tmp, n, 24, 8);\n    oracle_radix_pass_u32(tmp, out, n, 8, 8);"),
    # segmented scan that ignores the head flags
    "segscan_no_reset": ("            if (h[i])                                                                    \\\n                acc = (IDENT);",
                         "            if (0)                                                                       \\\n                acc = (IDENT);"),
    # segmented float64 sum that keeps the compensation across a head
    "segscan_f64_keeps_compensation": ("        if (h[i]) {\n            s = 0.0;\n            c = 0.0;\n        }",
                                       "        if (h[i]) {\n            s = 0.0;\n        }"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle._SRC).read()
    assert src.count(old) >= 1, "mutation anchor not found: " + name
    mutated = src.replace(old, new, 1)
    csrc = os.path.join(str(tmp_path), "oracle_mut.c")
    with open(csrc, "w") as f:
        f.write(mutated)
    so = oracle.build(force=True, src=csrc, out=os.path.join(str(tmp_path), "liboracle_mut.so"))
    mut = oracle.Oracle(oracle.load_library(so))
    caught = None
    for pin in ALL_PINS:
        try:
            pin(mut)
        except AssertionError:
            caught = pin.__name__
            break
    assert caught, "no pin caught mutant " + name
