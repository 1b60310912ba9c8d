"""Sequential CPU oracle for the device-wide scan and stream compaction.

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` import this package.  The product
library never loads it and has no CPU fallback.  The arithmetic lives in
``oracle.c`` (plain C loops, compiled with gcc, no CUDA headers); this module
only compiles it, loads it with ctypes and marshals numpy arrays.

What each function computes, and the passage it follows, is documented in
``oracle.c``.  Parity status: every function is pinned by the ``-m "not gpu"``
tests (page examples under ``tests/golden/``, closed forms, invariants,
library special cases, exhaustive brute force on short inputs); the float32
sum is pinned to the exactly rounded prefix sums (``math.fsum``) within the
fp64 error bound.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

PRED = {"gt": 0, "ge": 1, "lt": 2, "le": 3, "eq": 4, "ne": 5}

# (op, numpy dtype) -> (C function, dtype the bits are passed as): the
# operators whose result has the input's type.
_U32, _U64 = np.dtype(np.uint32), np.dtype(np.uint64)
_GENERIC = {}
for _op in ("prod", "and", "or", "xor"):
    for _dt in (np.int32, np.uint32):
        _GENERIC[(_op, np.dtype(_dt))] = "oracle_scan_%s_u32" % _op
    for _dt in (np.int64, np.uint64):
        _GENERIC[(_op, np.dtype(_dt))] = "oracle_scan_%s_u64" % _op
for _dt in (np.int64, np.uint64):
    _GENERIC[("sum", np.dtype(_dt))] = "oracle_scan_sum_u64"
for _op in ("max", "min"):
    for _dt, _sfx in ((np.uint32, "u32"), (np.int64, "i64"), (np.uint64, "u64"),
                      (np.float32, "f32"), (np.float64, "f64")):
        _GENERIC[(_op, np.dtype(_dt))] = "oracle_scan_%s_%s" % (_op, _sfx)
_GENERIC[("min", np.dtype(np.int32))] = "oracle_scan_min_i32"

# (op, numpy dtype) -> the segmented scan (head flags) of the same operator
_SEGMENTED = {k: v.replace("oracle_scan_", "oracle_segscan_") for k, v in _GENERIC.items()}
for _dt in (np.int32, np.uint32):
    _SEGMENTED[("sum", np.dtype(_dt))] = "oracle_segscan_sum_u32"
_SEGMENTED[("max", np.dtype(np.int32))] = "oracle_segscan_max_i32"
_SEGMENTED[("sum", np.dtype(np.float32))] = "oracle_segscan_sum_f32"
_SEGMENTED[("sum", np.dtype(np.float64))] = "oracle_segscan_sum_f64"


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile oracle.c into a shared library with gcc (-O2, no fast-math)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + ".tmp.%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                               "-fno-fast-math", "-ffp-contract=off", src, "-o", tmp, "-lm"])
        os.replace(tmp, out)
    return out


def load_library(path: str) -> ctypes.CDLL:
    """Load an oracle shared library and declare its signatures."""
    lib = ctypes.CDLL(path)
    P, I64, INT, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
    for name in ("oracle_scan_sum_u32", "oracle_scan_sum_f32", "oracle_scan_max_i32",
                 "oracle_scan_affine_u32"):
        f = getattr(lib, name)
        f.argtypes = [P, P, I64, INT]
        f.restype = None
    for name in ("oracle_scan_batched_sum_u32", "oracle_scan_batched_sum_f32",
                 "oracle_scan_batched_max_i32", "oracle_scan_batched_affine_u32"):
        f = getattr(lib, name)
        f.argtypes = [P, P, I64, I64, INT]
        f.restype = None
    for name in _GENERIC.values():
        f = getattr(lib, name)
        f.argtypes = [P, P, I64, INT]
        f.restype = None
    for name in ("oracle_scan_sum_f64", "oracle_scan_maxcount_i32"):
        f = getattr(lib, name)
        f.argtypes = [P, P, I64, INT]
        f.restype = None
    for name in set(_SEGMENTED.values()) | {"oracle_segscan_affine_u32", "oracle_segscan_maxcount_i32"}:
        f = getattr(lib, name)
        f.argtypes = [P, P, P, I64, INT]
        f.restype = None
    for name in ("oracle_compact_i32", "oracle_compact_u32", "oracle_compact_f32"):
        f = getattr(lib, name)
        f.argtypes = [P, I64, INT, D, P]
        f.restype = I64
    for name in ("oracle_abs_prefix_f32", "oracle_abs_prefix_f64"):
        f = getattr(lib, name)
        f.argtypes = [P, P, I64]
        f.restype = None
    lib.oracle_radix_pass_u32.argtypes = [P, P, I64, INT, INT]
    lib.oracle_radix_pass_u32.restype = None
    lib.oracle_radix_sort_u32.argtypes = [P, P, P, I64]
    lib.oracle_radix_sort_u32.restype = None
    lib.oracle_histogram.argtypes = [P, I64, I64, P]
    lib.oracle_histogram.restype = I64
    lib.oracle_bin_offsets.argtypes = [P, I64, I64, P, P]
    lib.oracle_bin_offsets.restype = I64
    return lib


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
        return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


class Oracle:
    """numpy-level wrapper around one loaded oracle library."""

    def __init__(self, cdll: ctypes.CDLL):
        self.c = cdll

    # -- scans ---------------------------------------------------------------
    def scan(self, x: np.ndarray, op: str, exclusive: bool) -> np.ndarray:
        """Inclusive or exclusive scan of a 1-D array.

        op: "sum" (int32/uint32/int64/uint64 -> same dtype, wrapping; float32 ->
            float64; float64 -> float64, compensated), "max" / "min" (int32,
            uint32, int64, uint64, float32, float64; floats propagate NaN),
            "prod" / "and" / "or" / "xor" (the four integer dtypes, wrapping),
            "affine" (uint32 array of shape (n, 2): rows (a, b)), "maxcount"
            (int32/uint32 array of shape (n, 2): rows (value, count)).
        """
        ex = 1 if exclusive else 0
        if op == "sum" and x.dtype in (np.int32, np.uint32):
            xs = np.ascontiguousarray(x).view(np.uint32)
            y = np.empty_like(xs)
            self.c.oracle_scan_sum_u32(_ptr(xs), _ptr(y), xs.size, ex)
            return y.view(x.dtype)
        if op == "sum" and x.dtype == np.float32:
            xs = np.ascontiguousarray(x)
            y = np.empty(xs.size, dtype=np.float64)
            self.c.oracle_scan_sum_f32(_ptr(xs), _ptr(y), xs.size, ex)
            return y
        if op == "max" and x.dtype == np.int32:
            xs = np.ascontiguousarray(x)
            y = np.empty_like(xs)
            self.c.oracle_scan_max_i32(_ptr(xs), _ptr(y), xs.size, ex)
            return y
        if op == "affine" and x.dtype == np.uint32 and x.ndim == 2 and x.shape[1] == 2:
            xs = np.ascontiguousarray(x)
            y = np.empty_like(xs)
            self.c.oracle_scan_affine_u32(_ptr(xs), _ptr(y), xs.shape[0], ex)
            return y
        if op == "sum" and x.dtype == np.float64:
            xs = np.ascontiguousarray(x)
            y = np.empty_like(xs)
            self.c.oracle_scan_sum_f64(_ptr(xs), _ptr(y), xs.size, ex)
            return y
        if op == "maxcount" and x.dtype in (np.int32, np.uint32) and x.ndim == 2 and x.shape[1] == 2:
            xs = np.ascontiguousarray(x).view(np.uint32)
            y = np.empty_like(xs)
            self.c.oracle_scan_maxcount_i32(_ptr(xs), _ptr(y), xs.shape[0], ex)
            return y.view(x.dtype)
        name = _GENERIC.get((op, x.dtype))
        if name is not None and x.ndim == 1:
            xs = np.ascontiguousarray(x)
            y = np.empty_like(xs)
            getattr(self.c, name)(_ptr(xs), _ptr(y), xs.size, ex)
            return y
        raise ValueError("unsupported oracle scan: op=%s dtype=%s shape=%s" % (op, x.dtype, x.shape))

    def scan_batched(self, x: np.ndarray, op: str, exclusive: bool) -> np.ndarray:
        """Row-wise scans of a row-major (rows, cols) matrix ((rows, cols, 2) for affine)."""
        ex = 1 if exclusive else 0
        rows, cols = x.shape[0], x.shape[1]
        if op == "sum" and x.dtype in (np.int32, np.uint32):
            xs = np.ascontiguousarray(x).view(np.uint32)
            y = np.empty_like(xs)
            self.c.oracle_scan_batched_sum_u32(_ptr(xs), _ptr(y), rows, cols, ex)
            return y.view(x.dtype)
        if op == "sum" and x.dtype == np.float32:
            xs = np.ascontiguousarray(x)
            y = np.empty(xs.shape, dtype=np.float64)
            self.c.oracle_scan_batched_sum_f32(_ptr(xs), _ptr(y), rows, cols, ex)
            return y
        if op == "max" and x.dtype == np.int32:
            xs = np.ascontiguousarray(x)
            y = np.empty_like(xs)
            self.c.oracle_scan_batched_max_i32(_ptr(xs), _ptr(y), rows, cols, ex)
            return y
        if op == "affine" and x.dtype == np.uint32 and x.ndim == 3 and x.shape[2] == 2:
            xs = np.ascontiguousarray(x)
            y = np.empty_like(xs)
            self.c.oracle_scan_batched_affine_u32(_ptr(xs), _ptr(y), rows, cols, ex)
            return y
        # every other operator (its result has the input's type): the 1-D
        # oracle on each row
        xs = np.ascontiguousarray(x)
        if rows == 0:
            return np.empty_like(xs)
        return np.stack([self.scan(xs[r], op, exclusive) for r in range(rows)])

    def scan_segmented(self, x: np.ndarray, heads: np.ndarray, op: str, exclusive: bool) -> np.ndarray:
        """Segmented scan: heads[i] != 0 starts a new segment at i (element 0
        always starts one); the same operators and dtypes as scan()."""
        ex = 1 if exclusive else 0
        h = np.ascontiguousarray(heads, dtype=np.uint8)
        n = x.shape[0]
        if h.shape != (n,):
            raise ValueError("heads must hold one flag per element")
        if op in ("affine", "maxcount") and x.ndim == 2 and x.shape[1] == 2 and x.dtype in (np.int32, np.uint32):
            xs = np.ascontiguousarray(x).view(np.uint32)
            y = np.empty_like(xs)
            getattr(self.c, "oracle_segscan_%s_i32" % op if op == "maxcount" else "oracle_segscan_affine_u32")(
                _ptr(xs), _ptr(h), _ptr(y), n, ex)
            return y.view(x.dtype)
        name = _SEGMENTED.get((op, x.dtype))
        if name is None or x.ndim != 1:
            raise ValueError("unsupported oracle segmented scan: op=%s dtype=%s" % (op, x.dtype))
        xs = np.ascontiguousarray(x)
        if x.dtype in (np.int32, np.uint32) and "u32" in name:
            xs = xs.view(np.uint32)
        elif x.dtype in (np.int64, np.uint64) and "u64" in name:
            xs = xs.view(np.uint64)
        y = np.empty(n, dtype=np.float64) if x.dtype == np.float32 and op == "sum" else np.empty_like(xs)
        getattr(self.c, name)(_ptr(xs), _ptr(h), _ptr(y), n, ex)
        return y if y.dtype == np.float64 and x.dtype == np.float32 else y.view(x.dtype)

    # -- histogram and bin offsets ------------------------------------------
    def histogram(self, bins: np.ndarray, nbins: int):
        """(counts int64[nbins], entries outside [0, nbins))."""
        b = np.ascontiguousarray(bins, dtype=np.int32)
        counts = np.empty(max(nbins, 0), dtype=np.int64)
        outside = self.c.oracle_histogram(_ptr(b), b.size, nbins, _ptr(counts))
        return counts, int(outside)

    def bin_offsets(self, bins: np.ndarray, nbins: int):
        """(offsets int64[nbins + 1], entries outside [0, nbins)): the exclusive
        scan of the histogram, the number of counted entries last (COO row
        indices -> CSR row offsets)."""
        b = np.ascontiguousarray(bins, dtype=np.int32)
        counts = np.empty(max(nbins, 0), dtype=np.int64)
        offsets = np.empty(nbins + 1, dtype=np.int64)
        outside = self.c.oracle_bin_offsets(_ptr(b), b.size, nbins, _ptr(counts), _ptr(offsets))
        return offsets, int(outside)

    # -- radix sort ------------------------------------------------------------
    def radix_pass(self, keys: np.ndarray, shift: int, bits: int) -> np.ndarray:
        """One stable counting-sort pass of uint32 keys by (k >> shift) & (2^bits - 1), 1 <= bits <= 8."""
        if not (1 <= bits <= 8 and 0 <= shift <= 31):
            raise ValueError("bits in [1, 8], shift in [0, 31]")
        k = np.ascontiguousarray(keys, dtype=np.uint32)
        out = np.empty_like(k)
        self.c.oracle_radix_pass_u32(_ptr(k), _ptr(out), k.size, shift, bits)
        return out

    def radix_sort(self, keys: np.ndarray) -> np.ndarray:
        """uint32 keys sorted ascending by four 8-bit passes."""
        k = np.ascontiguousarray(keys, dtype=np.uint32)
        out = np.empty_like(k)
        tmp = np.empty_like(k)
        self.c.oracle_radix_sort_u32(_ptr(k), _ptr(out), _ptr(tmp), k.size)
        return out

    # -- compaction ----------------------------------------------------------
    def compact(self, x: np.ndarray, pred: str, threshold: float):
        """Order-preserving compaction; returns (kept values, count)."""
        xs = np.ascontiguousarray(x)
        out = np.empty_like(xs)
        fn = {np.dtype(np.int32): self.c.oracle_compact_i32,
              np.dtype(np.uint32): self.c.oracle_compact_u32,
              np.dtype(np.float32): self.c.oracle_compact_f32}.get(xs.dtype)
        if fn is None:
            raise ValueError("unsupported oracle compaction dtype %s" % xs.dtype)
        cnt = fn(_ptr(xs), xs.size, PRED[pred], float(threshold), _ptr(out))
        return out[:cnt].copy(), int(cnt)

    def abs_prefix(self, x: np.ndarray) -> np.ndarray:
        """s[i] = |x[0]| + ... + |x[i]| in fp64 (scale of the float tolerances)."""
        if x.dtype == np.float64:
            xs = np.ascontiguousarray(x)
            s = np.empty(xs.size, dtype=np.float64)
            self.c.oracle_abs_prefix_f64(_ptr(xs), _ptr(s), xs.size)
            return s
        xs = np.ascontiguousarray(x, dtype=np.float32)
        s = np.empty(xs.size, dtype=np.float64)
        self.c.oracle_abs_prefix_f32(_ptr(xs), _ptr(s), xs.size)
        return s


_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(lib())
    return _default


def scan(x, op, exclusive):
    return default().scan(x, op, exclusive)


def scan_batched(x, op, exclusive):
    return default().scan_batched(x, op, exclusive)


def scan_segmented(x, heads, op, exclusive):
    return default().scan_segmented(x, heads, op, exclusive)


def compact(x, pred, threshold):
    return default().compact(x, pred, threshold)


def histogram(bins, nbins):
    return default().histogram(bins, nbins)


def radix_pass(keys, shift, bits):
    return default().radix_pass(keys, shift, bits)


def radix_sort(keys):
    return default().radix_sort(keys)


def bin_offsets(bins, nbins):
    return default().bin_offsets(bins, nbins)


def abs_prefix(x):
    return default().abs_prefix(x)
