"""sc_release_stream gives back the device memory the library keeps per stream.

A stream that ran a device scan holds a look-back workspace (at least 1 MiB),
and one that ran sc_scan_host also holds three 64 MiB staging buffers.  After
sc_release_stream the device's free memory is back where it started, for 50
streams in a row; a released stream works again on its next call.
"""
import numpy as np
import pytest

import oracle
from gpu_helpers import ensure_lib
import stream_compaction_gb300 as sc

pytestmark = pytest.mark.gpu

MiB = 1 << 20


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _use_stream(s, x, y, hx, hy, n):
    """One device scan and one host-buffer scan on stream s."""
    sp = int(s.cuda_stream)
    assert sc.sc_scan_exclusive(sc.SC_U32, sc.SC_SUM, x.data_ptr(), y.data_ptr(), n, sp) == sc.SC_OK
    assert sc.sc_scan_host(sc.SC_U32, sc.SC_SUM, 1, hx.data_ptr(), hy.data_ptr(), n, sp) == sc.SC_OK
    assert sc.sc_get_device_error(sp) == sc.SC_OK


def test_release_returns_memory():
    import torch
    n = (1 << 20) + 3
    xh = np.random.default_rng(3).integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
    x = torch.from_numpy(xh.view(np.int32)).cuda()
    y = torch.empty_like(x)
    hx = torch.from_numpy(xh.view(np.int32)).pin_memory()
    hy = torch.empty_like(hx).pin_memory()
    want = oracle.scan(xh, "sum", True)
    streams = [torch.cuda.Stream() for _ in range(50)]
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]

    # a stream in use holds its workspace and staging buffers ...
    _use_stream(streams[0], x, y, hx, hy, n)
    held = free0 - torch.cuda.mem_get_info()[0]
    assert held >= 3 * 64 * MiB, held
    # ... until it is released
    assert sc.sc_release_stream(int(streams[0].cuda_stream)) == sc.SC_OK
    assert torch.cuda.mem_get_info()[0] >= free0 - 8 * MiB

    for s in streams:
        _use_stream(s, x, y, hx, hy, n)
        assert np.array_equal(hy.numpy().view(np.uint32), want)
        assert sc.sc_release_stream(int(s.cuda_stream)) == sc.SC_OK
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] >= free0 - 8 * MiB

    # released streams work again, and releasing an unused stream is a no-op
    _use_stream(streams[1], x, y, hx, hy, n)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), want)
    assert sc.sc_release_stream(int(streams[1].cuda_stream)) == sc.SC_OK
    assert sc.sc_release_stream(int(streams[2].cuda_stream)) == sc.SC_OK
