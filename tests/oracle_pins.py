"""Pins for the CPU oracle: checks against what the pages and the mathematics fix.

Each ``pin_*`` function takes an ``oracle.Oracle`` instance and raises
AssertionError if it disagrees with:
  * the worked examples the pages print (fixtures under tests/golden/, each
    with its citation);
  * closed forms (all ones, x[i] = i, all 0xFFFFFFFF, affine special cases);
  * invariants (exclusive = inclusive shifted right with the identity in
    front; the last inclusive value is the reduction; compaction count is the
    flag sum, order kept);
  * library routines that compute the same thing a different way
    (numpy.cumsum with uint32 wraparound, numpy.maximum.accumulate, boolean
    mask selection, math.fsum);
  * brute force over every input of length <= 8 (<= 5 or 6 for the added
    operators) on small alphabets, against a divide-and-conquer fold (a
    different association order than the oracle's left-to-right loop) or, for
    affine maps, against applying the maps one after another to a point, and
    for (max, count) pairs against the definition (largest value, total count
    of its occurrences).

The same functions run against deliberately broken copies of the oracle
(tests/test_oracle_mutants.py) to show that each plausible mistake is caught.
"""
from __future__ import annotations

import itertools
import math

import numpy as np

from conftest import load_golden

M32 = 1 << 32
INT32_MIN = -(1 << 31)
INT32_MAX = (1 << 31) - 1


# ------------------------------------------------------------------ helpers
def _all_sequences(alphabet, length):
    """Every sequence of `length` symbols from `alphabet`, as a (k, length) array."""
    if length == 0:
        return np.zeros((1, 0), dtype=np.asarray(alphabet).dtype)
    idx = np.array(list(itertools.product(range(len(alphabet)), repeat=length)), dtype=np.int64)
    return np.asarray(alphabet)[idx]


def _dc_fold(cols, op, identity):
    """Divide-and-conquer fold over a list of column arrays (keeps left-to-right order)."""
    if len(cols) == 0:
        return identity
    if len(cols) == 1:
        return cols[0]
    mid = len(cols) // 2
    return op(_dc_fold(cols[:mid], op, identity), _dc_fold(cols[mid:], op, identity))


def _apply_affine(a, b, h):
    return (a.astype(np.uint64) * np.uint64(h) + b.astype(np.uint64)) % np.uint64(M32)


# ------------------------------------------------------------ page examples
def pin_golden_sum_examples(o):
    for name in ("l7_sum_example.txt", "l7_sandwich.txt"):
        g = load_golden(name)
        x = np.array(g["input"], dtype=np.int32)
        assert o.scan(x, "sum", False).tolist() == g["inclusive"], name
        assert o.scan(x, "sum", True).tolist() == g["exclusive"], name
        assert o.scan(x.view(np.uint32), "sum", True).tolist() == g["exclusive"], name
        yf = o.scan(x.astype(np.float32), "sum", False)
        assert yf.tolist() == [float(v) for v in g["inclusive"]], name
        if "left_over" in g:
            assert g["length"][0] - int(o.scan(x, "sum", False)[-1]) == g["left_over"][0]
    g = load_golden("tut_flag_positions.txt")
    assert o.scan(np.array(g["input"], dtype=np.int32), "sum", True).tolist() == g["exclusive"]
    g = load_golden("pmpp_ch9_examples.txt")
    x5 = np.array(g["sum5_input"], dtype=np.int32)
    assert o.scan(x5, "sum", False).tolist() == g["sum5_inclusive"]
    assert o.scan(x5, "sum", True).tolist() == g["sum5_exclusive"]
    x8 = np.array(g["sum8_input"], dtype=np.int32)
    assert o.scan(x8, "sum", True).tolist() == g["sum8_exclusive"]
    assert int(o.scan(x8, "sum", False)[-1]) == g["sum8_total"][0]


def pin_golden_compaction_examples(o):
    for name, pfx in (("l7_compaction.txt", ""), ("pmpp_ch9_examples.txt", "filter_")):
        g = load_golden(name)
        x = np.array(g[pfx + "input"], dtype=np.int32)
        pred, thr = g[pfx + "pred"][0], g[pfx + "threshold"][0]
        out, cnt = o.compact(x, pred, thr)
        assert out.tolist() == g[pfx + "output"], name
        assert cnt == sum(g[pfx + "flags"]) == len(g[pfx + "output"]), name
        flags = np.array(g[pfx + "flags"], dtype=np.int32)
        assert o.scan(flags, "sum", True).tolist() == g[pfx + "flag_exclusive_scan"], name
        # the scatter: kept element i goes to slot exclusive_scan(flags)[i]
        pos = o.scan(flags, "sum", True)
        scattered = [None] * cnt
        for i in range(x.size):
            if flags[i]:
                scattered[pos[i]] = int(x[i])
        assert scattered == out.tolist(), name
        # same compaction on float32 and uint32-representable data
        outf, cntf = o.compact(x.astype(np.float32), pred, thr)
        assert outf.tolist() == [float(v) for v in g[pfx + "output"]] and cntf == cnt


def pin_golden_identities(o):
    g = load_golden("pmpp_ch9_identities.txt")
    for x in (np.array([5, 7], dtype=np.int32), np.array([-3], dtype=np.int32)):
        assert int(o.scan(x, "sum", True)[0]) == g["sum"][0]
        assert int(o.scan(x, "max", True)[0]) == g["max_i32"][0]
    assert float(o.scan(np.array([2.5], dtype=np.float32), "sum", True)[0]) == float(g["sum"][0])
    # exclusive affine starts with the map that leaves every point unchanged
    ab = np.array([[3, 4], [5, 6]], dtype=np.uint32)
    y = o.scan(ab, "affine", True)
    for h in (0, 1, 12345, M32 - 1):
        assert int(_apply_affine(y[:1, 0], y[:1, 1], h)[0]) == h
    # empty inputs
    for op, x in (("sum", np.zeros(0, np.int32)), ("max", np.zeros(0, np.int32)),
                  ("sum", np.zeros(0, np.float32)), ("affine", np.zeros((0, 2), np.uint32))):
        assert o.scan(x, op, True).shape[0] == 0 and o.scan(x, op, False).shape[0] == 0
    out, cnt = o.compact(np.zeros(0, np.int32), "gt", 0)
    assert cnt == 0 and out.size == 0


# -------------------------------------------------------------- closed forms
def pin_closed_forms(o):
    for n in (1, 2, 7, 1000, 1 << 17):
        i = np.arange(n, dtype=np.uint64)
        ones = np.ones(n, dtype=np.uint32)
        assert np.array_equal(o.scan(ones, "sum", True), i.astype(np.uint32))
        assert np.array_equal(o.scan(ones, "sum", False), (i + 1).astype(np.uint32))
        assert np.array_equal(o.scan(np.ones(n, np.float32), "sum", True), i.astype(np.float64))
        # x[i] = i  ->  inclusive i(i+1)/2 mod 2^32
        xi = i.astype(np.uint32)
        tri = ((i * (i + np.uint64(1))) // np.uint64(2)) % np.uint64(M32)
        assert np.array_equal(o.scan(xi, "sum", False), tri.astype(np.uint32))
        # all 0xFFFFFFFF -> inclusive -(i+1) mod 2^32
        allf = np.full(n, 0xFFFFFFFF, dtype=np.uint32)
        neg = (np.uint64(M32) - (i + np.uint64(1)) % np.uint64(M32)) % np.uint64(M32)
        assert np.array_equal(o.scan(allf, "sum", False), neg.astype(np.uint32))
        assert np.array_equal(o.scan(allf.view(np.int32), "sum", False),
                              (-(i.astype(np.int64) + 1)).astype(np.int32))
        # max over ascending input is the input; over descending it is x[0]
        asc = np.arange(n, dtype=np.int32) - n // 2
        assert np.array_equal(o.scan(asc, "max", False), asc)
        assert np.array_equal(o.scan(asc[::-1].copy(), "max", False), np.full(n, asc[-1], np.int32))


def pin_affine_special_cases(o):
    rng = np.random.default_rng(7)
    n = 5000
    b = rng.integers(0, M32, n, dtype=np.uint64).astype(np.uint32)
    a = rng.integers(0, M32, n, dtype=np.uint64).astype(np.uint32)
    # all a = 1: translations compose by adding; the result is (1, sum of b)
    y = o.scan(np.stack([np.ones(n, np.uint32), b], axis=1), "affine", False)
    assert np.all(y[:, 0] == 1)
    assert np.array_equal(y[:, 1], np.cumsum(b, dtype=np.uint32))
    # all b = 0: scalings compose by multiplying; the result is (prefix product, 0)
    y = o.scan(np.stack([a, np.zeros(n, np.uint32)], axis=1), "affine", False)
    assert np.all(y[:, 1] == 0)
    assert np.array_equal(y[:, 0], (np.cumprod(a.astype(np.uint64)) % np.uint64(M32)).astype(np.uint32))


# ---------------------------------------------------------------- invariants
def _random_inputs():
    rng = np.random.default_rng(12345)
    n = 30011
    return {
        "sum_i32": rng.integers(-1000, 1000, n).astype(np.int32),
        "sum_u32": rng.integers(0, M32, n, dtype=np.uint64).astype(np.uint32),
        "max_i32": rng.integers(INT32_MIN, INT32_MAX, n, endpoint=True).astype(np.int32),
        "affine": rng.integers(0, M32, (n, 2), dtype=np.uint64).astype(np.uint32),
        "sum_f32": rng.uniform(-1, 1, n).astype(np.float32),
    }


def pin_invariants(o):
    d = _random_inputs()
    for key, op in (("sum_i32", "sum"), ("sum_u32", "sum"), ("max_i32", "max"),
                    ("affine", "affine"), ("sum_f32", "sum")):
        x = d[key]
        inc = o.scan(x, op, False)
        exc = o.scan(x, op, True)
        ident = {"sum": 0, "max": INT32_MIN}.get(op)
        # exclusive = inclusive shifted right by one with the identity in front
        assert np.array_equal(exc[1:], inc[:-1]), key
        if op == "affine":
            assert exc[0].tolist() == [1, 0]
        else:
            assert exc[0] == ident, key
        # the last inclusive value is the reduction of the whole array
        if op == "sum" and x.dtype != np.float32:
            assert int(inc[-1]) % M32 == int(x.astype(np.int64).sum()) % M32, key
        elif op == "max":
            assert int(inc[-1]) == int(x.max())
        elif op == "sum":
            assert abs(float(inc[-1]) - math.fsum(x.astype(np.float64))) <= 1e-9
    # max-scan is monotone and each output is one of the inputs seen so far
    x = d["max_i32"]
    y = o.scan(x, "max", False)
    assert np.all(np.diff(y.astype(np.int64)) >= 0)
    assert np.all(y >= x)
    for i in range(0, x.size, 997):
        assert int(y[i]) in set(x[:i + 1].tolist())


def pin_affine_recurrence(o):
    """y[i] applied to h[-1] equals the sequential recurrence h[i] = a[i]*h[i-1] + b[i]."""
    x = _random_inputs()["affine"][:4000]
    inc = o.scan(x, "affine", False)
    exc = o.scan(x, "affine", True)
    for h0 in (0, 1, 0xDEADBEEF, M32 - 1):
        h = h0
        hs = []
        for a, b in x.tolist():
            hs.append(h)
            h = (a * h + b) % M32
            hs[-1] = (hs[-1], h)
        before = np.array([p for p, _ in hs], dtype=np.uint64)
        after = np.array([q for _, q in hs], dtype=np.uint64)
        assert np.array_equal(_apply_affine(inc[:, 0], inc[:, 1], h0), after)
        assert np.array_equal(_apply_affine(exc[:, 0], exc[:, 1], h0), before)


# ------------------------------------------------------ library special cases
def pin_library_special_cases(o):
    d = _random_inputs()
    x = d["sum_u32"]
    assert np.array_equal(o.scan(x, "sum", False), np.cumsum(x, dtype=np.uint32))
    xi = d["sum_i32"]
    assert np.array_equal(o.scan(xi, "sum", False), np.cumsum(xi, dtype=np.int32))
    xm = d["max_i32"]
    assert np.array_equal(o.scan(xm, "max", False), np.maximum.accumulate(xm))
    assert o.scan(xm[:3000], "max", False).tolist() == list(itertools.accumulate(xm[:3000].tolist(), max))
    # compaction equals boolean-mask selection, for every predicate
    for dt, x in ((np.int32, d["sum_i32"]), (np.uint32, d["sum_u32"]), (np.float32, d["sum_f32"])):
        for pred, fn in (("gt", np.greater), ("ge", np.greater_equal), ("lt", np.less),
                         ("le", np.less_equal), ("eq", np.equal), ("ne", np.not_equal)):
            for thr in (0, 0.5, -3, float(x[17])):
                out, cnt = o.compact(x, pred, thr)
                mask = fn(x.astype(np.float64), thr)
                assert cnt == int(mask.sum()), (dt, pred, thr)
                assert np.array_equal(out, x[mask]), (dt, pred, thr)


def pin_float_fp64_accumulation(o):
    """The float32 sum is the fp64 running sum: within n*2^-53*sum|x| of the exact prefix."""
    rng = np.random.default_rng(99)
    x = rng.uniform(-1, 1, 3000).astype(np.float32)
    y = o.scan(x, "sum", False)
    ye = o.scan(x, "sum", True)
    xs = x.astype(np.float64).tolist()
    s = o.abs_prefix(x)
    for i in range(0, x.size, 7):
        exact = math.fsum(xs[:i + 1])
        assert abs(y[i] - exact) <= (i + 1) * 2.0 ** -53 * s[i] + 1e-300, i
        assert abs(ye[i] - math.fsum(xs[:i])) <= (i + 1) * 2.0 ** -53 * s[i] + 1e-300, i
        assert abs(s[i] - math.fsum(abs(v) for v in xs[:i + 1])) <= (i + 1) * 2.0 ** -53 * s[i]
    # small terms that float32 accumulation would lose are kept
    tiny = np.full(1 << 12, 2.0 ** -30, dtype=np.float32)
    z = o.scan(np.concatenate([np.ones(1, np.float32), tiny]), "sum", False)
    assert z[-1] == 1.0 + tiny.size * 2.0 ** -30


# ------------------------------------------------------ batched row scans
def pin_batched_rows(o):
    d = _random_inputs()
    for key, op in (("sum_i32", "sum"), ("max_i32", "max"), ("sum_f32", "sum")):
        x = d[key][:30000].reshape(120, 250)
        for ex in (False, True):
            yb = o.scan_batched(x, op, ex)
            for r in (0, 1, 77, 119):
                assert np.array_equal(yb[r], o.scan(x[r].copy(), op, ex)), (key, ex, r)
    xa = d["affine"][:30000].reshape(120, 250, 2)
    for ex in (False, True):
        yb = o.scan_batched(xa, "affine", ex)
        for r in (0, 5, 119):
            assert np.array_equal(yb[r], o.scan(xa[r].copy(), "affine", ex))
    # row independence: each row starts from the identity
    x = np.ones((64, 33), dtype=np.int32)
    assert np.array_equal(o.scan_batched(x, "sum", True), np.tile(np.arange(33, dtype=np.int32), (64, 1)))


# ------------------------------------------------------------- brute force
def _brute_scan(o, alphabet, op_name, op, identity, max_len=8):
    for length in range(0, max_len + 1):
        seqs = _all_sequences(alphabet, length)
        for ex in (False, True):
            if length == 0:
                assert o.scan(seqs[0], op_name, ex).size == 0
                continue
            got = o.scan_batched(seqs, op_name, ex)
            cols = [seqs[:, j] for j in range(length)]
            for i in range(length):
                pre = cols[:i] if ex else cols[:i + 1]
                want = _dc_fold(pre, op, identity)
                if np.isscalar(want) or np.ndim(want) == 0:
                    want = np.full(seqs.shape[0], want)
                assert np.array_equal(got[:, i].astype(np.int64), np.asarray(want).astype(np.int64)), \
                    (op_name, length, ex, i)
            # the 1-D entry point agrees with the batched one on a sample of rows
            for r in range(0, seqs.shape[0], max(1, seqs.shape[0] // 50)):
                assert np.array_equal(o.scan(seqs[r].copy(), op_name, ex), got[r])


def pin_brute_force_sum(o):
    add = lambda p, q: (p.astype(np.int64) + q.astype(np.int64)) % M32
    _brute_scan(o, np.array([0, 1, 2], dtype=np.uint32), "sum", add, 0)
    _brute_scan(o, np.array([0xFFFFFFFF, 1, 0x80000000], dtype=np.uint32), "sum", add, 0, max_len=7)


def pin_brute_force_max(o):
    mx = lambda p, q: np.maximum(p.astype(np.int64), q.astype(np.int64))
    _brute_scan(o, np.array([INT32_MIN, -1, 0, 1, INT32_MAX], dtype=np.int32), "max", mx, INT32_MIN)


def pin_brute_force_affine(o):
    """Every sequence of <= 8 maps from a 4-map alphabet: y[i] must act on a point
    as the maps x[0], ..., x[i] applied one after another."""
    alphabet = np.array([[0, 0], [1, 1], [2, 3], [0xFFFFFFFF, 5]], dtype=np.uint32)
    for length in range(1, 9):
        idx = _all_sequences(np.arange(4), length)
        seqs = alphabet[idx]                       # (k, length, 2)
        for ex in (False, True):
            got = o.scan_batched(seqs, "affine", ex)
            for h0 in (0, 1):                     # a map a*h+b is fixed by its values at 0 and 1
                h = np.full(seqs.shape[0], h0, dtype=np.uint64)
                for i in range(length):
                    nxt = _apply_affine(seqs[:, i, 0], seqs[:, i, 1], h)
                    want = h if ex else nxt
                    assert np.array_equal(_apply_affine(got[:, i, 0], got[:, i, 1], h0), want), \
                        (length, ex, i, h0)
                    h = nxt


def pin_brute_force_compaction(o):
    for length in range(0, 9):
        seqs = _all_sequences(np.array([-1, 0, 1], dtype=np.int32), length)
        for pred, fn in (("gt", lambda v, t: v > t), ("ge", lambda v, t: v >= t),
                         ("lt", lambda v, t: v < t), ("le", lambda v, t: v <= t),
                         ("eq", lambda v, t: v == t), ("ne", lambda v, t: v != t)):
            for thr in (0, -1, 0.5):
                for r in range(seqs.shape[0]):
                    row = seqs[r]
                    out, cnt = o.compact(row, pred, thr)
                    want = [v for v in row.tolist() if fn(v, thr)]
                    assert out.tolist() == want and cnt == len(want), (row.tolist(), pred, thr)


# ------------------------------------- more operators and element types
M64 = 1 << 64
INT64_MIN = -(1 << 63)
INT64_MAX = (1 << 63) - 1


def _fmax_first(p, q):
    """max propagating NaN, the earlier of equal values kept (vectorised)."""
    return np.where(np.isnan(p), p, np.where(np.isnan(q), q, np.where(q > p, q, p)))


def _fmin_first(p, q):
    return np.where(np.isnan(p), p, np.where(np.isnan(q), q, np.where(q < p, q, p)))


def _same_float(a, b):
    """Equal bit for bit, or both NaN."""
    a, b = np.asarray(a), np.asarray(b)
    bits = np.uint32 if a.dtype == np.float32 else np.uint64
    return bool(np.all((a.view(bits) == b.view(bits)) | (np.isnan(a) & np.isnan(b))))


def pin_golden_identities_more(o):
    g = load_golden("pmpp_ch9_identities.txt")
    for dt in (np.int32, np.uint32, np.int64, np.uint64):
        x = np.array([5, 7, 2], dtype=dt)
        assert int(o.scan(x, "prod", True)[0]) == g["prod"][0], dt
        assert int(o.scan(x, "or", True)[0]) == g["or"][0], dt
        assert int(o.scan(x, "xor", True)[0]) == 0, dt
    assert int(o.scan(np.array([5, 7], np.int32), "min", True)[0]) == g["min_i32"][0]
    assert int(o.scan(np.array([5, 7], np.uint32), "and", True)[0]) == g["and_u32"][0]
    assert int(o.scan(np.array([5, 7], np.uint64), "and", True)[0]) == M64 - 1
    assert int(o.scan(np.array([5, 7], np.int32), "and", True)[0]) == -1
    # the integer infinities are the extremes of each type
    for dt, lo, hi in ((np.uint32, 0, M32 - 1), (np.int64, INT64_MIN, INT64_MAX), (np.uint64, 0, M64 - 1)):
        x = np.array([5, 7], dtype=dt)
        assert int(o.scan(x, "max", True)[0]) == lo and int(o.scan(x, "min", True)[0]) == hi, dt
    for dt in (np.float32, np.float64):
        x = np.array([2.5, -1.0], dtype=dt)
        assert o.scan(x, "max", True)[0] == float(g["max_float"][0])
        assert o.scan(x, "min", True)[0] == float(g["min_float"][0])
    assert float(o.scan(np.array([2.5], np.float64), "sum", True)[0]) == float(g["sum"][0])
    yv = o.scan(np.array([[5, 1], [6, 2]], dtype=np.int32), "maxcount", True)
    assert yv[0].tolist() == [g["max_i32"][0], 0]
    for op, x in (("prod", np.zeros(0, np.uint64)), ("min", np.zeros(0, np.float64)),
                  ("sum", np.zeros(0, np.float64)), ("maxcount", np.zeros((0, 2), np.int32))):
        assert o.scan(x, op, True).shape[0] == 0 and o.scan(x, op, False).shape[0] == 0


def pin_closed_forms_more(o):
    for n in (1, 2, 5, 33, 70, 1000):
        i = np.arange(n, dtype=np.int64)
        # prod of all 3s: 3^(i+1) modulo 2^32 and 2^64
        p32 = [pow(3, k + 1, M32) for k in range(n)]
        p64 = [pow(3, k + 1, M64) for k in range(n)]
        assert o.scan(np.full(n, 3, np.uint32), "prod", False).tolist() == p32
        assert o.scan(np.full(n, 3, np.uint64), "prod", False).tolist() == p64
        # prod of 1..n: the factorials modulo 2^64
        fact, f = [], 1
        for k in range(1, n + 1):
            f = f * k % M64
            fact.append(f)
        assert o.scan(np.arange(1, n + 1, dtype=np.uint64), "prod", False).tolist() == fact
        # or of 1 << (i mod 32): 2^(i+1) - 1 until all 32 bits are set
        x = (np.uint64(1) << (i % 32).astype(np.uint64)).astype(np.uint32)
        want = [min((1 << (k + 1)) - 1, M32 - 1) for k in range(n)]
        assert o.scan(x, "or", False).tolist() == want
        # and of all-ones-but-bit (i mod 32): bits 0..i cleared
        assert o.scan(~x, "and", False).tolist() == [(M32 - 1) ^ w for w in want]
        # xor of 0..i: i, 1, i+1, 0 by i mod 4
        xr = [(k, 1, k + 1, 0)[k % 4] for k in range(n)]
        assert o.scan(i.astype(np.uint32), "xor", False).tolist() == xr
        assert o.scan(i.astype(np.uint64), "xor", False).tolist() == xr
        # 64-bit sums: x[i] = i -> i(i+1)/2; all ones-complement -> -(i+1) mod 2^64
        assert o.scan(i.astype(np.uint64), "sum", False).tolist() == [k * (k + 1) // 2 for k in range(n)]
        assert o.scan(np.full(n, M64 - 1, np.uint64), "sum", False).tolist() == [(M64 - k - 1) % M64
                                                                                    for k in range(n)]
        assert o.scan(np.full(n, -1, np.int64), "sum", True).tolist() == [-k for k in range(n)]
        # min over descending input is the input, over ascending it is x[0]
        for dt in (np.int32, np.uint32, np.int64, np.uint64, np.float32, np.float64):
            asc = np.arange(n).astype(dt)
            assert np.array_equal(o.scan(asc[::-1].copy(), "min", False), asc[::-1])
            assert np.array_equal(o.scan(asc, "min", False), np.zeros(n, dt))
            assert np.array_equal(o.scan(asc, "max", False), asc)
        # float64 sum of ones: the exact integers
        assert o.scan(np.ones(n), "sum", True).tolist() == [float(k) for k in range(n)]
        # (max, count) of equal values counts them; of rising values keeps count 1
        eq = np.stack([np.full(n, 7, np.int32), np.ones(n, np.int32)], axis=1)
        assert o.scan(eq, "maxcount", False).tolist() == [[7, k + 1] for k in range(n)]
        up = np.stack([np.arange(n, dtype=np.int32), np.ones(n, np.int32)], axis=1)
        assert o.scan(up, "maxcount", False).tolist() == [[k, 1] for k in range(n)]


def _more_inputs():
    rng = np.random.default_rng(2024)
    n = 20011
    u32 = rng.integers(0, M32, n, dtype=np.uint64).astype(np.uint32)
    u64 = rng.integers(0, M64, n, dtype=np.uint64)
    f64 = rng.uniform(-1, 1, n) * 10.0 ** rng.integers(-8, 8, n)
    return {"u32": u32, "i32": u32.view(np.int32), "u64": u64, "i64": u64.view(np.int64),
            "f32": rng.uniform(-3, 3, n).astype(np.float32), "f64": f64}


def pin_library_special_cases_more(o):
    d = _more_inputs()
    for key in ("u32", "i32", "u64", "i64"):
        x = d[key]
        dt = x.dtype
        assert np.array_equal(o.scan(x, "max", False), np.maximum.accumulate(x)), key
        assert np.array_equal(o.scan(x, "min", False), np.minimum.accumulate(x)), key
        assert np.array_equal(o.scan(x, "and", False), np.bitwise_and.accumulate(x)), key
        assert np.array_equal(o.scan(x, "or", False), np.bitwise_or.accumulate(x)), key
        assert np.array_equal(o.scan(x, "xor", False), np.bitwise_xor.accumulate(x)), key
        assert np.array_equal(o.scan(x, "prod", False), np.cumprod(x, dtype=dt)), key
        if dt.itemsize == 8:
            assert np.array_equal(o.scan(x, "sum", False), np.cumsum(x, dtype=dt)), key
    for key in ("f32", "f64"):
        x = d[key].copy()
        x[[3, 700, 701, 9000]] = np.nan
        lo = np.array([-np.inf], dtype=x.dtype)
        hi = np.array([np.inf], dtype=x.dtype)
        assert _same_float(o.scan(x, "max", False), np.maximum.accumulate(np.concatenate([lo, x]))[1:]), key
        assert _same_float(o.scan(x, "min", False), np.minimum.accumulate(np.concatenate([hi, x]))[1:]), key
        assert np.isnan(o.scan(x, "max", False)[3:]).all() and not np.isnan(o.scan(x, "max", False)[:3]).any()
    # (max, count) with unit counts: the running max and how often it has occurred so far
    v = (d["u32"] % np.uint32(50)).astype(np.int32)
    y = o.scan(np.stack([v, np.ones_like(v)], axis=1), "maxcount", False)
    run = np.maximum.accumulate(v)
    assert np.array_equal(y[:, 0], run)
    for i in range(0, v.size, 613):
        assert int(y[i, 1]) == int(np.count_nonzero(v[:i + 1] == run[i])), i


def pin_float64_sum(o):
    """The float64 sum is within a few units in the last place of the exactly
    rounded prefix sum (math.fsum), far inside the fp64 scan error bound."""
    x = _more_inputs()["f64"][:4000]
    xs = x.tolist()
    y, ye = o.scan(x, "sum", False), o.scan(x, "sum", True)
    s = o.abs_prefix(x)
    for i in range(0, x.size, 5):
        exact = math.fsum(xs[:i + 1])
        assert abs(y[i] - exact) <= 4 * 2.0 ** -53 * abs(exact) + 1e-28 * s[i], i
        assert abs(ye[i] - math.fsum(xs[:i])) <= 4 * 2.0 ** -53 * abs(math.fsum(xs[:i])) + 1e-28 * s[i], i
        assert abs(s[i] - math.fsum(abs(v) for v in xs[:i + 1])) <= (i + 1) * 2.0 ** -53 * s[i]
    # cancellation that a plain running fp64 sum gets wrong
    z = o.scan(np.array([1.0, 1e100, 1.0, -1e100]), "sum", False)
    assert z[-1] == 2.0


def _brute_scan_bits(o, alphabet, op_name, op, identity, max_len=5, floats=False):
    """Like _brute_scan, with outputs compared bit for bit (floats: NaN = NaN)."""
    for length in range(0, max_len + 1):
        seqs = _all_sequences(alphabet, length)
        for ex in (False, True):
            if length == 0:
                assert o.scan(seqs[0], op_name, ex).size == 0
                continue
            got = o.scan_batched(seqs, op_name, ex)
            cols = [seqs[:, j] for j in range(length)]
            for i in range(length):
                pre = cols[:i] if ex else cols[:i + 1]
                want = _dc_fold(pre, op, identity)
                want = np.broadcast_to(np.asarray(want, dtype=seqs.dtype), (seqs.shape[0],))
                if floats:
                    assert _same_float(got[:, i], want), (op_name, length, ex, i)
                else:
                    assert np.array_equal(got[:, i], want), (op_name, length, ex, i)


def pin_brute_force_more(o):
    with np.errstate(over="ignore"):
        u32 = np.array([0, 1, 2, 0x80000000, 0xFFFFFFFF], dtype=np.uint32)
        u64 = np.array([0, 1, 3, 1 << 63, M64 - 1], dtype=np.uint64)
        for alphabet in (u32, u64):
            dt = alphabet.dtype
            ones = np.array(np.iinfo(dt).max, dtype=dt)
            _brute_scan_bits(o, alphabet, "prod", lambda p, q: (p * q).astype(dt), np.array(1, dt))
            _brute_scan_bits(o, alphabet, "and", lambda p, q: p & q, ones)
            _brute_scan_bits(o, alphabet, "or", lambda p, q: p | q, np.array(0, dt))
            _brute_scan_bits(o, alphabet, "xor", lambda p, q: p ^ q, np.array(0, dt))
            _brute_scan_bits(o, alphabet, "max", np.maximum, np.array(0, dt))
            _brute_scan_bits(o, alphabet, "min", np.minimum, ones)
            if dt == np.uint64:
                _brute_scan_bits(o, alphabet, "sum", lambda p, q: (p + q).astype(dt), np.array(0, dt))
        for alphabet in (u32.view(np.int32), u64.view(np.int64)):
            dt = alphabet.dtype
            info = np.iinfo(dt)
            _brute_scan_bits(o, alphabet, "max", np.maximum, np.array(info.min, dt))
            _brute_scan_bits(o, alphabet, "min", np.minimum, np.array(info.max, dt))
        for dt in (np.float32, np.float64):
            fl = np.array([np.nan, -np.inf, -0.0, 0.0, 1.5, np.inf], dtype=dt)
            _brute_scan_bits(o, fl, "max", _fmax_first, np.array(-np.inf, dt), floats=True)
            _brute_scan_bits(o, fl, "min", _fmin_first, np.array(np.inf, dt), floats=True)
    # (max, count) pairs: every sequence of <= 6 pairs from a 4-pair alphabet
    alphabet = np.array([[1 << 31, 1], [0, 1], [0, 2], [5, 0xFFFFFFFF]], dtype=np.uint32)  # value bits: INT32_MIN, 0, 0, 5
    for length in range(1, 7):
        seqs = alphabet[_all_sequences(np.arange(4), length)]          # (k, length, 2)
        for ex in (False, True):
            got = o.scan_batched(seqs, "maxcount", ex)
            v = seqs[:, :, 0].view(np.int32).astype(np.int64)
            c = seqs[:, :, 1].astype(np.int64)
            for i in range(length):
                m = i if ex else i + 1
                if m == 0:
                    wv, wc = np.full(seqs.shape[0], INT32_MIN), np.zeros(seqs.shape[0], np.int64)
                else:
                    wv = v[:, :m].max(axis=1)
                    wc = np.where(v[:, :m] == wv[:, None], c[:, :m], 0).sum(axis=1) % M32
                assert np.array_equal(got[:, i, 0].view(np.int32).astype(np.int64), wv), (length, ex, i)
                assert np.array_equal(got[:, i, 1].astype(np.int64), wc), (length, ex, i)


# ------------------------------------------------------------ segmented scans
_SEG_CASES = [("i32", "sum"), ("u32", "sum"), ("i32", "max"), ("f32", "sum"), ("u32", "prod"), ("i32", "and"),
              ("u32", "or"), ("u32", "xor"), ("i32", "min"), ("u32", "max"), ("u32", "min"), ("u64", "sum"),
              ("i64", "prod"), ("u64", "and"), ("i64", "or"), ("u64", "xor"), ("i64", "max"), ("i64", "min"),
              ("u64", "max"), ("u64", "min"), ("f32", "max"), ("f32", "min"), ("f64", "sum"), ("f64", "max"),
              ("f64", "min"), ("affine", "affine"), ("maxcount", "maxcount")]


def _seg_input(kind, n, rng):
    if kind in ("affine", "maxcount"):
        v = rng.integers(0, 1 << 32, (n, 2), dtype=np.uint64).astype(np.uint32)
        if kind == "maxcount":
            v[:, 0] = rng.integers(-3, 3, n).astype(np.int32).view(np.uint32)
            v[:, 1] = rng.integers(0, 3, n)
        return v
    if kind in ("f32", "f64"):
        x = rng.uniform(-5, 5, n).astype(np.float32 if kind == "f32" else np.float64)
        x[rng.integers(0, n, max(1, n // 50))] = np.nan
        return x
    dt = {"i32": np.int32, "u32": np.uint32, "i64": np.int64, "u64": np.uint64}[kind]
    return rng.integers(0, 1 << 62, n, dtype=np.int64).astype(np.uint64).astype(np.dtype(dt).str.replace("i", "u"))\
        .view(dt) | np.array(1, dt)


def _seg_equal(a, b):
    if a.dtype.kind == "f":
        return _same_float(a, b) if a.dtype == b.dtype else np.array_equal(a, b)
    return np.array_equal(a, b)


def pin_segmented_is_scan_per_segment(o):
    """The segmented scan equals the plain scan of each segment on its own."""
    rng = np.random.default_rng(31)
    n = 3001
    for kind, op in _SEG_CASES:
        x = _seg_input(kind, n, rng)
        for density in (0.0, 0.003, 0.05, 0.5):
            h = (rng.random(n) < density).astype(np.uint8)
            starts = [0] + [i for i in range(1, n) if h[i]]
            ends = starts[1:] + [n]
            for ex in (False, True):
                y = o.scan_segmented(x, h, op, ex)
                want = np.concatenate([o.scan(x[a:b].copy(), op, ex) for a, b in zip(starts, ends)])
                assert _seg_equal(y, want), (kind, op, density, ex)


def pin_segmented_special_cases(o):
    rng = np.random.default_rng(32)
    n = 2000
    for kind, op in _SEG_CASES:
        x = _seg_input(kind, n, rng)
        none = np.zeros(n, np.uint8)
        allh = np.ones(n, np.uint8)
        for ex in (False, True):
            assert _seg_equal(o.scan_segmented(x, none, op, ex), o.scan(x, op, ex)), (kind, op, ex)
        # every element its own segment: inclusive gives x, exclusive the identity everywhere
        inc = o.scan_segmented(x, allh, op, False)
        exc = o.scan_segmented(x, allh, op, True)
        if op == "sum" and kind == "f32":
            assert np.array_equal(inc, x.astype(np.float64), equal_nan=True)
        else:
            assert _seg_equal(inc, x), (kind, op)
        first = o.scan(x[:1].copy(), op, True)
        assert _seg_equal(exc, np.repeat(first, n, axis=0)), (kind, op)
    # heads at multiples of cols: the batched row scans
    d = _random_inputs()
    x = d["sum_i32"][:30000]
    h = np.zeros(30000, np.uint8)
    h[::250] = 1
    for ex in (False, True):
        assert np.array_equal(o.scan_segmented(x, h, "sum", ex), o.scan_batched(x.reshape(120, 250), "sum", ex).ravel())


def pin_segmented_brute_force(o):
    """Every head pattern of every input of length <= 6 on a small alphabet."""
    for length in range(1, 7):
        seqs = _all_sequences(np.array([0, 1, 5], dtype=np.uint32), length)
        for mask in range(1 << length):
            h = np.array([(mask >> j) & 1 for j in range(length)], dtype=np.uint8)
            for r in range(0, seqs.shape[0], 7):
                row = seqs[r]
                for ex in (False, True):
                    got = o.scan_segmented(row, h, "sum", ex).tolist()
                    want, acc = [], 0
                    for j in range(length):
                        if h[j]:
                            acc = 0
                        if ex:
                            want.append(acc)
                            acc = acc + int(row[j])
                        else:
                            acc = acc + int(row[j])
                            want.append(acc)
                    assert got == want, (row.tolist(), h.tolist(), ex)


def pin_segmented_first_satisfying(o):
    """The pages' use of a max scan: the first element of each segment that
    satisfies a predicate is where the predicate holds and the exclusive
    segmented max of the predicate is still 0."""
    rng = np.random.default_rng(33)
    n = 5000
    p = (rng.random(n) < 0.2).astype(np.int32)
    h = (rng.random(n) < 0.01).astype(np.uint8)
    seen = o.scan_segmented(p, h, "max", True)
    first = (p == 1) & (seen <= 0)
    want, found = [], False
    for i in range(n):
        if i == 0 or h[i]:
            found = False
        want.append(bool(p[i]) and not found)
        found = found or bool(p[i])
    assert first.tolist() == want


# ------------------------------------------------- histogram and bin offsets
def pin_histogram_and_bin_offsets(o):
    rng = np.random.default_rng(41)
    for n, nbins in ((0, 5), (1, 1), (1000, 7), (50000, 256), (30011, 100000)):
        bins = rng.integers(-3, nbins + 3, n).astype(np.int32)
        counts, outside = o.histogram(bins, nbins)
        inside = bins[(bins >= 0) & (bins < nbins)]
        # numpy's bincount is the same histogram computed another way
        assert np.array_equal(counts, np.bincount(inside, minlength=nbins).astype(np.int64))
        assert outside == n - inside.size
        offsets, outside2 = o.bin_offsets(bins, nbins)
        assert outside2 == outside and offsets.size == nbins + 1
        assert offsets[0] == 0 and offsets[-1] == inside.size
        assert np.array_equal(np.diff(offsets), counts)
        # for sorted bins the offsets are where each bin starts (searchsorted), the CSR row pointers
        srt = np.sort(inside)
        assert np.array_equal(offsets, np.searchsorted(srt, np.arange(nbins + 1), side="left"))
    # the pages' radix-sort use: bucket starts are the exclusive scan of the digit histogram
    keys = rng.integers(0, 1 << 32, 20000, dtype=np.uint64).astype(np.uint32)
    digit = (keys >> np.uint32(8)) & np.uint32(255)
    starts, _ = o.bin_offsets(digit.astype(np.int32), 256)
    order = np.argsort(digit, kind="stable")
    sd = digit[order]
    for d in (0, 17, 255):
        hit = np.flatnonzero(sd == d)
        if hit.size:
            assert hit[0] == starts[d] and hit[-1] == starts[d + 1] - 1
    # COO -> CSR on a small matrix written out by hand: rows of the entries, 4 rows
    rows = np.array([0, 0, 1, 3, 3, 3], dtype=np.int32)
    assert o.bin_offsets(rows, 4)[0].tolist() == [0, 2, 3, 3, 6]


# ----------------------------------------------------------------- radix sort
def pin_radix_pass_and_sort(o):
    rng = np.random.default_rng(51)
    for n in (0, 1, 2, 17, 1000, 65537):
        keys = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
        keys[: n // 3] &= np.uint32(0x00FF00FF)          # repeated digits
        for shift, bits in ((0, 8), (8, 8), (24, 8), (3, 5), (31, 1), (28, 4)):
            got = o.radix_pass(keys, shift, bits)
            digit = (keys >> np.uint32(shift)) & np.uint32((1 << bits) - 1)
            # a stable partition by the digit is numpy's stable argsort of the digits
            assert np.array_equal(got, keys[np.argsort(digit, kind="stable")]), (n, shift, bits)
        # four 8-bit passes sort the keys
        assert np.array_equal(o.radix_sort(keys), np.sort(keys)), n
    # stability, by hand: equal digits keep their input order
    keys = np.array([0x102, 0x001, 0x201, 0x002, 0x101], dtype=np.uint32)
    assert o.radix_pass(keys, 0, 8).tolist() == [0x001, 0x201, 0x101, 0x102, 0x002]
    assert o.radix_pass(keys, 8, 8).tolist() == [0x001, 0x002, 0x102, 0x101, 0x201]


ALL_PINS = [
    pin_golden_sum_examples, pin_golden_compaction_examples, pin_golden_identities,
    pin_closed_forms, pin_affine_special_cases, pin_invariants, pin_affine_recurrence,
    pin_library_special_cases, pin_float_fp64_accumulation, pin_batched_rows,
    pin_brute_force_sum, pin_brute_force_max, pin_brute_force_affine, pin_brute_force_compaction,
    pin_golden_identities_more, pin_closed_forms_more, pin_library_special_cases_more, pin_float64_sum,
    pin_brute_force_more, pin_segmented_is_scan_per_segment, pin_segmented_special_cases,
    pin_segmented_brute_force, pin_segmented_first_satisfying, pin_histogram_and_bin_offsets,
    pin_radix_pass_and_sort,
]
