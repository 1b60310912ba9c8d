"""sc_scan_noalloc: the single-pass scan with its workspace in a fixed device
array, for callers that cannot allocate device memory.

Its results must equal those of the allocating entry points (bit for bit for
integer, max and affine scans; within the float32 tolerance of the other
tests for float sums) on two calls in a row, since every call reuses the
same array.  This file is collected last so that a run stopping at the first
failure has already run every other test; it also passes alone in a fresh
process.
"""
import numpy as np
import pytest

from gpu_helpers import CODE, OPC, dev_buffer, ensure_lib, stream, to_device, to_host
import oracle
import stream_compaction_gb300 as sc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _inputs(kind, n, seed):
    rng = np.random.default_rng(seed)
    if kind == "u32":
        return rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32), "sum"
    if kind == "i32":
        return rng.integers(-1000, 1000, n).astype(np.int32), "sum"
    if kind == "max":
        return rng.integers(-(1 << 31), (1 << 31) - 1, n, endpoint=True).astype(np.int32), "max"
    if kind == "f32":
        return rng.uniform(-1, 1, n).astype(np.float32), "sum"
    return rng.integers(0, 1 << 32, (n, 2), dtype=np.uint64).astype(np.uint32), "affine"


def _run(fn_noalloc: bool, x, op, exclusive):
    n = x.shape[0]
    kind = "affine" if op == "affine" else {np.dtype(np.int32): "i32", np.dtype(np.uint32): "u32",
                                            np.dtype(np.float32): "f32"}[x.dtype]
    _, xin = to_device(x)
    _, xout = dev_buffer(xin.numel(), xin.dtype)
    if fn_noalloc:
        st = sc.sc_scan_noalloc(CODE[kind], OPC[op], int(exclusive), xin.data_ptr(), xout.data_ptr(), n, stream())
    elif exclusive:
        st = sc.sc_scan_exclusive(CODE[kind], OPC[op], xin.data_ptr(), xout.data_ptr(), n, stream())
    else:
        st = sc.sc_scan_inclusive(CODE[kind], OPC[op], xin.data_ptr(), xout.data_ptr(), n, stream())
    assert st == sc.SC_OK, sc.status_string(st)
    return to_host(xout, x)


@pytest.mark.parametrize("kind", ["u32", "i32", "max", "f32", "affine"])
@pytest.mark.parametrize("exclusive", [False, True])
def test_noalloc_matches_allocating_path_twice(kind, exclusive):
    for call, n in enumerate((3 * 4096 + 5, (1 << 20) + 17)):   # two calls in a row
        x, op = _inputs(kind, n, seed=call * 17 + len(kind))
        got = _run(True, x, op, exclusive)
        want = _run(False, x, op, exclusive)
        if kind == "f32":
            bound = 1e-5 * oracle.abs_prefix(x)
            assert np.all(np.abs(got.astype(np.float64) - want.astype(np.float64)) <= bound), call
        else:
            assert np.array_equal(got, want), call


def test_noalloc_full_capacity_and_limits():
    """At the limit every status slot of the fixed array is in use: seeded
    full-range uint32 input, every output against the oracle, on two calls in
    a row (the second reuses the array the first left behind)."""
    from stream_compaction_gb300 import synth
    n = sc.SC_NOALLOC_MAX_N
    for call in range(2):
        x = synth.full_u32_np(n, seed=20 + call)
        got = _run(True, x, "sum", call == 0)
        assert np.array_equal(got, oracle.scan(x, "sum", call == 0)), call
    # beyond the fixed scratch: refused before any launch
    assert sc.sc_scan_noalloc(sc.SC_U32, sc.SC_SUM, 1, 0x1000, 0x1000, n + 1, stream()) == sc.SC_ERR_WORKSPACE
    assert sc.sc_scan_noalloc(sc.SC_U32, sc.SC_SUM, 1, 0, 0, 0, stream()) == sc.SC_OK
    assert sc.sc_scan_noalloc(sc.SC_F32, sc.SC_MAX, 1, 0, 0, 0, stream()) == sc.SC_ERR_UNSUPPORTED


@pytest.mark.parametrize("kind", ["u32", "f32", "affine"])
@pytest.mark.parametrize("exclusive", [False, True])
def test_noalloc_unaligned_and_in_place(kind, exclusive):
    """Element-aligned (not 16-byte aligned) buffers take the kernel's
    partial-tile loads; in == out scans in place; both against the oracle."""
    n = 5 * 4096 + 77
    x, op = _inputs(kind, n, seed=31 + exclusive)
    ref = oracle.scan(x, op, exclusive)
    code = CODE["affine" if kind == "affine" else kind]
    off = 2 if kind == "affine" else 1
    for offset, inplace in ((off, False), (0, True), (off, True)):
        _, xin = to_device(x, offset)
        if inplace:
            xout = xin
        else:
            _, xout = dev_buffer(xin.numel(), xin.dtype, offset + 2)
        st = sc.sc_scan_noalloc(code, OPC[op], int(exclusive), xin.data_ptr(), xout.data_ptr(), n, stream())
        assert st == sc.SC_OK, sc.status_string(st)
        got = to_host(xout, x)
        if kind == "f32":
            assert np.all(np.abs(got.astype(np.float64) - ref) <= 1e-5 * oracle.abs_prefix(x)), (offset, inplace)
        else:
            assert np.array_equal(got, ref), (offset, inplace)
    assert sc.sc_scan_noalloc_error(stream()) == sc.SC_OK


def test_noalloc_timeout_is_reported():
    """A tile that never publishes (test hook, 50 ms bound): its successors give
    up, the array's error word records it, sc_scan_noalloc_error reports and
    clears it, and the next call is exact again."""
    n = 64 * 4096
    x = np.ones(n, dtype=np.uint32)
    _, xin = to_device(x)
    _, xout = dev_buffer(n, xin.dtype)
    assert sc.sc_scan_noalloc_error(stream()) == sc.SC_OK
    assert sc.sc_debug_set_lookback(5, -1, 0, 50_000_000) == sc.SC_OK
    try:
        assert sc.sc_scan_noalloc(sc.SC_U32, sc.SC_SUM, 1, xin.data_ptr(), xout.data_ptr(), n, stream()) == sc.SC_OK
        assert sc.sc_scan_noalloc_error(stream()) == sc.SC_ERR_LOOKBACK_TIMEOUT
        assert sc.sc_scan_noalloc_error(stream()) == sc.SC_OK   # cleared by the first query
    finally:
        sc.sc_debug_set_lookback(-1, -1, 0, 0)
    for _ in range(2):
        assert sc.sc_scan_noalloc(sc.SC_U32, sc.SC_SUM, 1, xin.data_ptr(), xout.data_ptr(), n, stream()) == sc.SC_OK
        assert np.array_equal(to_host(xout, x), np.arange(n, dtype=np.uint32))
    assert sc.sc_scan_noalloc_error(stream()) == sc.SC_OK
