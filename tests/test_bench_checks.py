"""The checks bench.py applies to every output of its timed configurations
(the `parity` verdict of each `configs` entry): each accepts the oracle's
result and rejects a result with one planted mistake.  CPU only."""
import os
import sys

import numpy as np
import pytest

import oracle

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def _plant(y, i, delta=1):
    z = y.copy()
    flat = z.reshape(-1)
    flat[i] = flat[i] + np.array(delta).astype(flat.dtype)
    return z


@pytest.mark.parametrize("exclusive", [False, True])
def test_sum_u32_check(exclusive):
    rng = np.random.default_rng(1)
    x = rng.integers(0, 1 << 32, 5000, dtype=np.uint64).astype(np.uint32)  # wraps mod 2^32
    y = oracle.scan(x, "sum", exclusive)
    assert bench._check_sum_u32(x, y, exclusive)
    for i in (0, 1, 2500, 4999):
        assert not bench._check_sum_u32(x, _plant(y, i), exclusive), i


def test_max_i32_check():
    rng = np.random.default_rng(2)
    x = rng.integers(-(1 << 31), (1 << 31) - 1, 5000).astype(np.int32)
    y = oracle.scan(x, "max", False)
    assert bench._check_max_i32(x, y)
    # a value below the running maximum, and one above it
    assert not bench._check_max_i32(x, _plant(y, 3000, -1))
    z = y.copy()
    z[4000] = np.int32((1 << 31) - 1)
    assert not bench._check_max_i32(x, z)


def test_affine_check():
    rng = np.random.default_rng(3)
    x = rng.integers(0, 1 << 32, (3000, 2), dtype=np.uint64).astype(np.uint32)
    y = oracle.scan(x, "affine", False)
    assert bench._check_affine(x, y)
    for i in (0, 1, 2 * 1500, 2 * 1500 + 1, 5999):
        assert not bench._check_affine(x, _plant(y, i)), i
    # the composition order matters: the second output with the two maps
    # applied in the other order (b = a0 * b1 + b0 instead of a1 * b0 + b1) fails
    swapped = y.copy()
    with np.errstate(over="ignore"):
        swapped[1, 1] = np.uint32(x[0, 0]) * np.uint32(x[1, 1]) + np.uint32(x[0, 1])
    assert swapped[1, 1] != y[1, 1]
    assert not bench._check_affine(x, swapped)


def test_rows_exclusive_check():
    rng = np.random.default_rng(4)
    x = rng.integers(0, 256, (40, 33)).astype(np.int32)
    y = oracle.scan_batched(x, "sum", True)
    assert bench._check_rows_exclusive(x, y)
    assert not bench._check_rows_exclusive(x, _plant(y, 0))            # a row's first output
    assert not bench._check_rows_exclusive(x, _plant(y, 33 * 7 + 12))  # inside a row
    # a carry across rows (one scan over the whole matrix) fails
    assert not bench._check_rows_exclusive(x, oracle.scan(x.reshape(-1), "sum", True).reshape(40, 33))


@pytest.mark.parametrize("exclusive", [False, True])
def test_f32_error_ratio(exclusive):
    rng = np.random.default_rng(5)
    x = rng.uniform(-1, 1, 20000).astype(np.float32)
    y = oracle.scan(x, "sum", exclusive).astype(np.float32)
    assert bench._f32_error_ratio(x, y, exclusive) < 0.1
    z = y.copy()
    z[15000] += np.float32(1e-3 * np.sum(np.abs(x[:15001])))  # 100x the bound there
    assert bench._f32_error_ratio(x, z, exclusive) > 1.0
