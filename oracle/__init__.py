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
    for name in ("oracle_compact_i32", "oracle_compact_u32", "oracle_compact_f32"):
        f = getattr(lib, name)
        f.argtypes = [P, I64, INT, D, P]
        f.restype = I64
    lib.oracle_abs_prefix_f32.argtypes = [P, P, I64]
    lib.oracle_abs_prefix_f32.restype = None
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

        op: "sum" (int32/uint32 -> same dtype, wraps mod 2^32; float32 -> float64),
            "max" (int32), "affine" (uint32 array of shape (n, 2): rows (a, b)).
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
        raise ValueError("unsupported oracle batched scan: op=%s dtype=%s" % (op, x.dtype))

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
        """s[i] = |x[0]| + ... + |x[i]| in fp64 (scale of the float32 tolerance)."""
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


def compact(x, pred, threshold):
    return default().compact(x, pred, threshold)


def abs_prefix(x):
    return default().abs_prefix(x)
