"""Failure detection without a GPU fault: every look-back wait is bounded.

A test hook makes one tile never publish its status; its successors must give
up after the (short) timeout, poison their own status, record
SC_ERR_LOOKBACK_TIMEOUT in the device error word and exit.  Nothing traps and
nothing hangs; the context stays usable and the next call is exact again.
"""
import numpy as np
import pytest

import oracle
from gpu_helpers import ensure_lib, gpu_scan, stream, to_device, dev_buffer
import stream_compaction_gb300 as sc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()
    yield
    sc.sc_debug_set_lookback(-1, -1, 0, 0)


def _raw_scan(x, exclusive=True):
    _, xin = to_device(x)
    _, xout = dev_buffer(xin.numel(), xin.dtype)
    fn = sc.sc_scan_exclusive if exclusive else sc.sc_scan_inclusive
    st = fn(sc.SC_U32, sc.SC_SUM, xin.data_ptr(), xout.data_ptr(), x.size, stream())
    return st, xout


@pytest.mark.parametrize("tiles,stall", [(64, 5), (20000, 7), (300, 0)])
def test_stalled_tile_times_out(tiles, stall):
    x = np.ones(tiles * 4096, dtype=np.uint32)
    assert sc.sc_debug_set_lookback(stall, -1, 0, 50_000_000) == sc.SC_OK  # 50 ms bound
    try:
        st, _ = _raw_scan(x)
        assert st == sc.SC_OK  # the launch itself is fine
        err = sc.sc_get_device_error(stream())
        if stall < tiles - 1:
            assert err == sc.SC_ERR_LOOKBACK_TIMEOUT
        assert sc.sc_get_device_error(stream()) == sc.SC_OK  # cleared by the first read
    finally:
        sc.sc_debug_set_lookback(-1, -1, 0, 0)
    # the workspace and the context are usable again, and results are exact
    y = gpu_scan(x, "sum", True)
    assert np.array_equal(y, np.arange(x.size, dtype=np.uint32))


def test_stalled_tile_in_compaction_times_out():
    import torch
    n = 50 * 4096
    x = np.arange(n, dtype=np.int32) - n // 2
    _, xin = to_device(x)
    _, xout = dev_buffer(n, xin.dtype)
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
    sc.sc_debug_set_lookback(3, -1, 0, 50_000_000)
    try:
        assert sc.sc_compact_if(sc.SC_I32, xin.data_ptr(), xout.data_ptr(), cnt.data_ptr(), n, sc.SC_GT, 0.0,
                                stream()) == sc.SC_OK
        assert sc.sc_get_device_error(stream()) == sc.SC_ERR_LOOKBACK_TIMEOUT
    finally:
        sc.sc_debug_set_lookback(-1, -1, 0, 0)
    assert sc.sc_compact_if(sc.SC_I32, xin.data_ptr(), xout.data_ptr(), cnt.data_ptr(), n, sc.SC_GT, 0.0,
                            stream()) == sc.SC_OK
    assert sc.sc_get_device_error(stream()) == sc.SC_OK
    ref, rc = oracle.compact(x, "gt", 0)
    assert int(cnt.item()) == rc
    assert np.array_equal(xout[:rc].cpu().numpy(), ref)


@pytest.mark.parametrize("delay_tile", [0, 3, 31, 32, 33, 500])
def test_slow_tile_gives_exact_results(delay_tile):
    """One tile sleeps 2 ms before publishing: its successors wait, then walk long
    chains of aggregates.  Results stay exact."""
    n = 700 * 4096 + 123
    rng = np.random.default_rng(delay_tile)
    x = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
    sc.sc_debug_set_lookback(-1, delay_tile, 2_000_000, 0)
    try:
        for ex in (True, False):
            y = gpu_scan(x, "sum", ex)
            assert np.array_equal(y, oracle.scan(x, "sum", ex))
        xa = rng.integers(0, 1 << 32, (n // 2, 2), dtype=np.uint64).astype(np.uint32)
        assert np.array_equal(gpu_scan(xa, "affine", False), oracle.scan(xa, "affine", False))
    finally:
        sc.sc_debug_set_lookback(-1, -1, 0, 0)


def test_caller_workspace():
    import torch
    n = 10 * 4096 + 1
    x = np.ones(n, dtype=np.uint32)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        need = sc.sc_workspace_bytes(n)
        ws = torch.empty(need + 256, dtype=torch.uint8, device="cuda")
        base = (ws.data_ptr() + 255) // 256 * 256
        assert sc.sc_set_workspace(base, need, int(s.cuda_stream)) == sc.SC_OK
        y = gpu_scan(x, "sum", True)
        assert np.array_equal(y, np.arange(n, dtype=np.uint32))
        # a call that needs more than the bound workspace is refused
        big = np.ones(100 * 4096, dtype=np.uint32)
        st, _ = _raw_scan(big)
        assert st == sc.SC_ERR_WORKSPACE
        assert sc.sc_set_workspace(0, 0, int(s.cuda_stream)) == sc.SC_OK  # unbind
        y = gpu_scan(big, "sum", True)
        assert np.array_equal(y, np.arange(big.size, dtype=np.uint32))
    torch.cuda.synchronize()


def test_many_streams_are_independent():
    import torch
    streams = [torch.cuda.Stream() for _ in range(4)]
    rng = np.random.default_rng(3)
    xs = [rng.integers(0, 1 << 32, 300 * 4096 + k, dtype=np.uint64).astype(np.uint32) for k in range(4)]
    ins, outs = [], []
    for x, s in zip(xs, streams):
        with torch.cuda.stream(s):
            _, xi = to_device(x)
            _, xo = dev_buffer(x.size, xi.dtype)
            assert sc.sc_scan_exclusive(sc.SC_U32, sc.SC_SUM, xi.data_ptr(), xo.data_ptr(), x.size,
                                        int(s.cuda_stream)) == sc.SC_OK
            ins.append(xi)
            outs.append(xo)
    torch.cuda.synchronize()
    for x, o in zip(xs, outs):
        assert np.array_equal(o.cpu().numpy().view(np.uint32), oracle.scan(x, "sum", True))


def _raw_segscan(x, heads):
    import torch
    _, xin = to_device(x)
    _, xout = dev_buffer(xin.numel(), xin.dtype)
    h = torch.from_numpy(heads).cuda()
    st = sc.sc_scan_segmented(sc.SC_U32, sc.SC_SUM, 1, xin.data_ptr(), h.data_ptr(), xout.data_ptr(), x.size,
                              stream())
    return st, xout


@pytest.mark.parametrize("density", [0.0, 1e-3])
def test_stalled_chunk_in_segmented_scan_times_out(density):
    """The persistent segmented scan (8192-element tiles, 2-tile chunks): a chunk
    that never publishes makes its successor's look-back time out even when
    later chunks hold heads and publish their own prefixes at once."""
    n = 200 * 8192 + 77
    rng = np.random.default_rng(3)
    x = rng.integers(0, 100, n).astype(np.uint32)
    h = (rng.random(n) < density).astype(np.uint8)
    assert sc.sc_debug_set_lookback(10, -1, 0, 50_000_000) == sc.SC_OK  # chunk 5 never publishes
    try:
        st, _ = _raw_segscan(x, h)
        assert st == sc.SC_OK
        assert sc.sc_get_device_error(stream()) == sc.SC_ERR_LOOKBACK_TIMEOUT
    finally:
        sc.sc_debug_set_lookback(-1, -1, 0, 0)
    st, y = _raw_segscan(x, h)
    assert st == sc.SC_OK and sc.sc_get_device_error(stream()) == sc.SC_OK
    assert np.array_equal(y.cpu().numpy().view(np.uint32), oracle.scan_segmented(x, h, "sum", True))


@pytest.mark.parametrize("delay_tile", [0, 9, 64])
def test_slow_chunk_in_segmented_scan_gives_exact_results(delay_tile):
    n = 150 * 8192 + 5
    rng = np.random.default_rng(delay_tile + 1)
    x = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
    h = (rng.random(n) < 2e-5).astype(np.uint8)          # most chunks without a head: long chains
    sc.sc_debug_set_lookback(-1, delay_tile, 2_000_000, 0)
    try:
        st, y = _raw_segscan(x, h)
        assert st == sc.SC_OK and sc.sc_get_device_error(stream()) == sc.SC_OK
    finally:
        sc.sc_debug_set_lookback(-1, -1, 0, 0)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), oracle.scan_segmented(x, h, "sum", True))
