"""Seeded synthetic inputs, identical on the host (numpy) and on a device (torch).

This module holds no scan or compaction arithmetic: it only draws numbers.
Both the tests (for the oracle and for the CUDA path) and ``bench.py`` take
their inputs from here, so the two sides always see the same bytes.

Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) used as a counter-based generator.  Element
``i`` of stream ``seed`` is the first SplitMix64 output from the state
``key = seed * 2**32 + i + offset``:

    z = key + 0x9E3779B97F4A7C15          (mod 2**64)
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
    z = (z ^ (z >> 27)) * 0x94D049BB133111EB
    r = z ^ (z >> 31)

Mappings from the 64-bit draw ``r``:
  * integer uniform on the closed range [lo, hi]:  lo + (r mod (hi - lo + 1));
  * float32 uniform on [-1, 1):  (r >> 40) * 2**-23 - 1  (exact in float32);
  * full-range 32-bit words:  r >> 32;
  * affine pairs (a, b):  a = r >> 32, b = r & 0xFFFFFFFF;
  * full-range 64-bit words:  r;
  * float64 uniform on [-1, 1):  (r >> 11) * 2**-52 - 1  (exact in float64);
  * (value, count) pairs:  value = r mod 1024, count = 1;
  * segment head flags with mean segment length L:  1 if r mod L == 0, else 0;
  * COO row indices of a sparse matrix with rows sorted: row r holds
    1 + (r_r mod 63) entries (r_r the draw of row r), so 32 on average.
``offset`` selects a substream (2**40 for the second workload drawn from the
same seed).
"""
from __future__ import annotations

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
M1 = 0xBF58476D1CE4E5B9
M2 = 0x94D049BB133111EB
SUBSTREAM = 1 << 40


# ---------------------------------------------------------------- numpy (host)
def draws_np(n: int, seed: int, offset: int = 0, start: int = 0) -> np.ndarray:
    """uint64 draws r_i for i in [start, start + n)."""
    key = np.arange(start, start + n, dtype=np.uint64)
    key += np.uint64((seed << 32) + offset)
    with np.errstate(over="ignore"):
        z = key + np.uint64(GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(M1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(M2)
        z = z ^ (z >> np.uint64(31))
    return z


def uniform_int_np(n, lo, hi, seed, offset=0, dtype=np.int32):
    m = hi - lo + 1
    assert 0 < m <= 1 << 31
    r = draws_np(n, seed, offset)
    v = (r % np.uint64(m)).astype(np.int64) + lo
    return v.astype(dtype)


def uniform_pm1_f32_np(n, seed, offset=0):
    r = draws_np(n, seed, offset)
    k = (r >> np.uint64(40)).astype(np.float64)
    return (k * 2.0 ** -23 - 1.0).astype(np.float32)


def full_u32_np(n, seed, offset=0):
    return (draws_np(n, seed, offset) >> np.uint64(32)).astype(np.uint32)


def affine_pairs_np(n, seed, offset=0):
    r = draws_np(n, seed, offset)
    out = np.empty((n, 2), dtype=np.uint32)
    out[:, 0] = (r >> np.uint64(32)).astype(np.uint32)
    out[:, 1] = (r & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    return out


def full_u64_np(n, seed, offset=0):
    return draws_np(n, seed, offset)


def uniform_pm1_f64_np(n, seed, offset=0):
    k = (draws_np(n, seed, offset) >> np.uint64(11)).astype(np.float64)
    return k * 2.0 ** -52 - 1.0


def maxcount_pairs_np(n, seed, offset=0):
    out = np.ones((n, 2), dtype=np.int32)
    out[:, 0] = (draws_np(n, seed, offset) % np.uint64(1024)).astype(np.int32)
    return out


def head_flags_np(n, seed, offset=0, period=1024):
    return (draws_np(n, seed, offset) % np.uint64(period) == 0).astype(np.uint8)


def coo_rows_np(nrows, seed, offset=0):
    lengths = (draws_np(nrows, seed, offset) % np.uint64(63)).astype(np.int64) + 1
    return np.repeat(np.arange(nrows, dtype=np.int32), lengths)


# --------------------------------------------------------------- torch (device)
def _s64(c: int) -> int:
    """The int64 whose two's-complement bits equal the uint64 constant c."""
    return c - (1 << 64) if c >= 1 << 63 else c


def _lsr(z, k: int):
    """Logical right shift of int64 bit patterns."""
    return (z >> k) & ((1 << (64 - k)) - 1)


def draws_torch(n: int, seed: int, offset: int = 0, start: int = 0, device="cpu"):
    """int64 tensor holding the bit patterns of the uint64 draws r_i."""
    import torch
    z = torch.arange(start, start + n, dtype=torch.int64, device=device)
    z += _s64(((seed << 32) + offset + GAMMA) % (1 << 64))
    z = (z ^ _lsr(z, 30)) * _s64(M1)
    z = (z ^ _lsr(z, 27)) * _s64(M2)
    z = z ^ _lsr(z, 31)
    return z


def _chunked(n, fn, out, chunk=1 << 26):
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = fn(s, e - s)
    return out


def uniform_int_torch(n, lo, hi, seed, offset=0, device="cpu", dtype=None):
    import torch
    dtype = dtype or torch.int32
    m = hi - lo + 1
    assert 0 < m <= 1 << 31
    out = torch.empty(n, dtype=dtype, device=device)

    def f(s, c):
        r = draws_torch(c, seed, offset, s, device)
        # unsigned r mod m from the two 32-bit halves (exact in int64 since m <= 2^31)
        hi32 = _lsr(r, 32)
        lo32 = r & 0xFFFFFFFF
        v = ((hi32 % m) * ((1 << 32) % m) + lo32) % m
        return (v + lo).to(dtype)
    return _chunked(n, f, out)


def uniform_pm1_f32_torch(n, seed, offset=0, device="cpu"):
    import torch
    out = torch.empty(n, dtype=torch.float32, device=device)

    def f(s, c):
        k = _lsr(draws_torch(c, seed, offset, s, device), 40).to(torch.float64)
        return (k * 2.0 ** -23 - 1.0).to(torch.float32)
    return _chunked(n, f, out)


def _low32_as_i32(v):
    import torch
    v = v & 0xFFFFFFFF
    return torch.where(v >= (1 << 31), v - (1 << 32), v).to(torch.int32)


def full_u32_torch(n, seed, offset=0, device="cpu"):
    """Full-range 32-bit words, stored as int32 bit patterns."""
    import torch
    out = torch.empty(n, dtype=torch.int32, device=device)
    return _chunked(n, lambda s, c: _low32_as_i32(_lsr(draws_torch(c, seed, offset, s, device), 32)), out)


def affine_pairs_torch(n, seed, offset=0, device="cpu"):
    """(n, 2) int32 tensor of (a, b) bit patterns."""
    import torch
    out = torch.empty((n, 2), dtype=torch.int32, device=device)

    def f(s, c):
        r = draws_torch(c, seed, offset, s, device)
        return torch.stack([_low32_as_i32(_lsr(r, 32)), _low32_as_i32(r)], dim=1)
    return _chunked(n, f, out)


def full_u64_torch(n, seed, offset=0, device="cpu"):
    """Full-range 64-bit words, stored as int64 bit patterns."""
    import torch
    out = torch.empty(n, dtype=torch.int64, device=device)
    return _chunked(n, lambda s, c: draws_torch(c, seed, offset, s, device), out)


def uniform_pm1_f64_torch(n, seed, offset=0, device="cpu"):
    import torch
    out = torch.empty(n, dtype=torch.float64, device=device)
    return _chunked(n, lambda s, c: _lsr(draws_torch(c, seed, offset, s, device), 11).to(torch.float64) * 2.0 ** -52
                    - 1.0, out)


def maxcount_pairs_torch(n, seed, offset=0, device="cpu"):
    """(n, 2) int32 tensor of (value, 1) pairs."""
    import torch
    out = torch.ones((n, 2), dtype=torch.int32, device=device)

    def f(s, c):
        v = draws_torch(c, seed, offset, s, device) & 1023
        return torch.stack([v.to(torch.int32), torch.ones_like(v, dtype=torch.int32)], dim=1)
    return _chunked(n, f, out)


def head_flags_torch(n, seed, offset=0, period=1024, device="cpu"):
    """uint8 flags: 1 where a segment starts."""
    import torch
    out = torch.empty(n, dtype=torch.uint8, device=device)

    def f(s, c):
        r = draws_torch(c, seed, offset, s, device)
        # unsigned r mod period from the two 32-bit halves, as in uniform_int_torch
        v = ((_lsr(r, 32) % period) * ((1 << 32) % period) + (r & 0xFFFFFFFF)) % period
        return (v == 0).to(torch.uint8)
    return _chunked(n, f, out)


def coo_rows_torch(nrows, seed, offset=0, device="cpu"):
    import torch
    r = draws_torch(nrows, seed, offset, 0, device)
    lengths = ((_lsr(r, 32) % 63) * ((1 << 32) % 63) + (r & 0xFFFFFFFF)) % 63 + 1
    return torch.repeat_interleave(torch.arange(nrows, dtype=torch.int32, device=device), lengths)


# ------------------------------------------------------------- named workloads
# The benchmark workloads (sizes, distributions and seeds), as data: the five
# configurations of the headline metric, then one per family of added operators
# (op: the operator the benchmark runs on it).
WORKLOADS = {
    "int32_sum_n1048593": dict(kind="int", n=(1 << 20) + 17, lo=0, hi=9, seed=0, offset=0),
    "float32_exsum_n2^26": dict(kind="pm1", n=1 << 26, seed=1, offset=0),
    "int32_compact_gt0_n2^27": dict(kind="int", n=1 << 27, lo=-(1 << 20), hi=(1 << 20) - 1, seed=2, offset=0),
    "int32_max_n2^27": dict(kind="u32", n=1 << 27, seed=3, offset=0),
    "affine_u32_n2^26": dict(kind="affine", n=1 << 26, seed=3, offset=SUBSTREAM),
    "uint32_exsum_n2^30": dict(kind="u32", n=1 << 30, seed=4, offset=0),
    "int32_rows_65536x4096": dict(kind="int", n=65536 * 4096, lo=0, hi=255, seed=4, offset=SUBSTREAM),
    "int64_exsum_n2^27": dict(kind="u64", n=1 << 27, seed=5, offset=0, op="sum"),
    "float64_exsum_n2^26": dict(kind="pm1_f64", n=1 << 26, seed=6, offset=0, op="sum"),
    "int32_min_n2^27": dict(kind="u32", n=1 << 27, seed=5, offset=SUBSTREAM, op="min"),
    "uint32_xor_n2^27": dict(kind="u32", n=1 << 27, seed=7, offset=0, op="xor"),
    "float32_max_n2^26": dict(kind="pm1", n=1 << 26, seed=7, offset=SUBSTREAM, op="max"),
    "maxcount_i32_n2^26": dict(kind="maxcount", n=1 << 26, seed=8, offset=0, op="maxcount"),
    # segmented sum: values as the batched rows, heads with mean segment length 1024
    "int32_segsum_n2^27": dict(kind="int", n=1 << 27, lo=0, hi=255, seed=9, offset=0, op="sum",
                               heads=dict(seed=9, offset=SUBSTREAM, period=1024)),
    # the same heads over float32 values on [-1, 1)
    "float32_segsum_n2^27": dict(kind="pm1", n=1 << 27, seed=13, offset=0, op="sum",
                                 heads=dict(seed=9, offset=SUBSTREAM, period=1024)),
    # bin offsets: the CSR row offsets of a COO matrix with 2^22 sorted rows
    # (about 2^27 entries), and the start of each bucket of an 8-bit radix digit
    "csr_rows_2^22": dict(kind="coo_rows", nrows=1 << 22, seed=10, offset=0),
    "digit_bins_n2^27": dict(kind="int", n=1 << 27, lo=0, hi=255, seed=11, offset=0, nbins=256),
    # radix sort: full-range 32-bit keys
    "uint32_sort_n2^27": dict(kind="u32", n=1 << 27, seed=12, offset=0),
}


def make_heads_np(spec: dict, n: int | None = None):
    h = spec["heads"]
    return head_flags_np(spec["n"] if n is None else n, h["seed"], h["offset"], h["period"])


def make_heads_torch(spec: dict, n: int | None = None, device="cpu"):
    h = spec["heads"]
    return head_flags_torch(spec["n"] if n is None else n, h["seed"], h["offset"], h["period"], device)


def make_np(spec: dict, n: int | None = None):
    n = spec.get("n") if n is None else n
    k = spec["kind"]
    if k == "int":
        return uniform_int_np(n, spec["lo"], spec["hi"], spec["seed"], spec["offset"])
    if k == "pm1":
        return uniform_pm1_f32_np(n, spec["seed"], spec["offset"])
    if k == "u32":
        return full_u32_np(n, spec["seed"], spec["offset"])
    if k == "affine":
        return affine_pairs_np(n, spec["seed"], spec["offset"])
    if k == "u64":
        return full_u64_np(n, spec["seed"], spec["offset"])
    if k == "pm1_f64":
        return uniform_pm1_f64_np(n, spec["seed"], spec["offset"])
    if k == "maxcount":
        return maxcount_pairs_np(n, spec["seed"], spec["offset"])
    if k == "coo_rows":
        return coo_rows_np(spec["nrows"], spec["seed"], spec["offset"])
    raise ValueError(k)


def make_torch(spec: dict, n: int | None = None, device="cpu"):
    n = spec.get("n") if n is None else n
    k = spec["kind"]
    if k == "int":
        return uniform_int_torch(n, spec["lo"], spec["hi"], spec["seed"], spec["offset"], device)
    if k == "pm1":
        return uniform_pm1_f32_torch(n, spec["seed"], spec["offset"], device)
    if k == "u32":
        return full_u32_torch(n, spec["seed"], spec["offset"], device)
    if k == "affine":
        return affine_pairs_torch(n, spec["seed"], spec["offset"], device)
    if k == "u64":
        return full_u64_torch(n, spec["seed"], spec["offset"], device)
    if k == "pm1_f64":
        return uniform_pm1_f64_torch(n, spec["seed"], spec["offset"], device)
    if k == "maxcount":
        return maxcount_pairs_torch(n, spec["seed"], spec["offset"], device)
    if k == "coo_rows":
        return coo_rows_torch(spec["nrows"], spec["seed"], spec["offset"], device)
    raise ValueError(k)
