"""CUDA graph capture: calls that keep look-back state on the host (epoch and
tile-counter base) refuse a capturing stream with SC_ERR_UNSUPPORTED before
launching anything, and work normally afterwards; the histogram, which keeps
no such state, can be captured and replayed."""
import numpy as np
import pytest

import oracle
from gpu_helpers import ensure_lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def test_capture_is_refused_and_later_calls_work():
    import torch
    import stream_compaction_gb300 as sc
    n = 5 * 4096 + 3
    rng = np.random.default_rng(1)
    xh = rng.integers(-50, 50, n).astype(np.int32)
    x = torch.from_numpy(xh).cuda()
    y = torch.zeros_like(x)
    cnt = torch.zeros(1, dtype=torch.int64, device="cuda")
    bins = torch.from_numpy(rng.integers(0, 100, n).astype(np.int32)).cuda()
    offs = torch.zeros(101, dtype=torch.int64, device="cuda")
    keys, ko, kt = x.clone(), torch.zeros_like(x), torch.zeros_like(x)
    heads = torch.zeros(n, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    st = {}
    with torch.cuda.stream(s):
        g.capture_begin()
        try:
            sp = s.cuda_stream
            st["scan"] = sc.sc_scan_exclusive(sc.SC_I32, sc.SC_SUM, x.data_ptr(), y.data_ptr(), n, sp)
            st["batched"] = sc.sc_scan_batched(sc.SC_I32, sc.SC_SUM, 1, x.data_ptr(), y.data_ptr(), 1, n, sp)
            st["segmented"] = sc.sc_scan_segmented(sc.SC_I32, sc.SC_SUM, 1, x.data_ptr(), heads.data_ptr(),
                                                   y.data_ptr(), n, sp)
            st["compact"] = sc.sc_compact_if(sc.SC_I32, x.data_ptr(), y.data_ptr(), cnt.data_ptr(), n, sc.SC_GT,
                                             0.0, sp)
            st["noalloc"] = sc.sc_scan_noalloc(sc.SC_I32, sc.SC_SUM, 1, x.data_ptr(), y.data_ptr(), n, sp)
            st["bin_offsets"] = sc.sc_bin_offsets(bins.data_ptr(), n, 100, offs.data_ptr(), sp)
            st["radix_sort"] = sc.sc_radix_sort_u32(keys.data_ptr(), ko.data_ptr(), kt.data_ptr(), n, sp)
            st["radix_pass"] = sc.sc_radix_pass_u32(keys.data_ptr(), ko.data_ptr(), n, 0, 8, sp)
        finally:
            g.capture_end()
    assert all(v == sc.SC_ERR_UNSUPPORTED for v in st.values()), st
    # the same calls outside capture, on the same stream
    sp = s.cuda_stream
    assert sc.sc_scan_exclusive(sc.SC_I32, sc.SC_SUM, x.data_ptr(), y.data_ptr(), n, sp) == sc.SC_OK
    s.synchronize()
    assert np.array_equal(y.cpu().numpy(), oracle.scan(xh, "sum", True))
    assert sc.sc_bin_offsets(bins.data_ptr(), n, 100, offs.data_ptr(), sp) == sc.SC_OK
    s.synchronize()
    assert np.array_equal(offs.cpu().numpy(), oracle.bin_offsets(bins.cpu().numpy(), 100)[0])
    assert sc.sc_get_device_error(sp) == sc.SC_OK


def test_histogram_capture_and_replay():
    import torch
    import stream_compaction_gb300 as sc
    n, nbins = 3 * 4096 + 17, 37
    rng = np.random.default_rng(2)
    bh = rng.integers(-3, nbins + 3, n).astype(np.int32)        # some entries outside [0, nbins)
    bins = torch.from_numpy(bh).cuda()
    counts = torch.full((nbins,), 7, dtype=torch.int64, device="cuda")
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        g.capture_begin()
        try:
            st = sc.sc_histogram(bins.data_ptr(), n, nbins, counts.data_ptr(), s.cuda_stream)
        finally:
            g.capture_end()
    assert st == sc.SC_OK
    want = oracle.histogram(bh, nbins)[0]
    for _ in range(2):                                            # each replay recounts from zero
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(counts.cpu().numpy(), want)
