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
    n = sc.SC_NOALLOC_MAX_N
    x = np.ones(n, dtype=np.uint32)
    for _ in range(2):
        got = _run(True, x, "sum", True)
        assert got[0] == 0 and got[-1] == n - 1 and np.array_equal(got[:4096], np.arange(4096, dtype=np.uint32))
    # beyond the fixed scratch: refused before any launch
    assert sc.sc_scan_noalloc(sc.SC_U32, sc.SC_SUM, 1, 0x1000, 0x1000, n + 1, stream()) == sc.SC_ERR_WORKSPACE
    assert sc.sc_scan_noalloc(sc.SC_U32, sc.SC_SUM, 1, 0, 0, 0, stream()) == sc.SC_OK
    assert sc.sc_scan_noalloc(sc.SC_F32, sc.SC_MAX, 1, 0, 0, 0, stream()) == sc.SC_ERR_UNSUPPORTED
