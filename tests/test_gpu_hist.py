"""GPU parity: histogram and bin offsets (COO row indices -> CSR row offsets,
radix digit bucket starts) against the CPU oracle, exactly."""
import numpy as np
import pytest

import oracle
from gpu_helpers import ensure_lib, stream, to_device

pytestmark = pytest.mark.gpu

NBINS = [1, 7, 256, 4096, 8193, 32768, 32769, 100000, 1 << 22]
SIZES = [0, 1, 3, 4, 5, 1000, 100003, (1 << 20) + 17, 3 * (1 << 21) + 7]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def gpu_bins(bins, nbins, offsets, off=0):
    import torch
    import stream_compaction_gb300 as sc
    n = bins.size
    _, b = to_device(bins if n else np.zeros(1, np.int32), off)
    out = torch.full((nbins + (1 if offsets else 0) + 2,), -5, dtype=torch.int64, device="cuda")
    fn = sc.sc_bin_offsets if offsets else sc.sc_histogram
    st = fn(b.data_ptr(), n, nbins, out.data_ptr(), stream())
    assert st == sc.SC_OK, sc.status_string(st)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    assert o[-1] == -5 and o[-2] == -5               # nothing written past the end
    return o[:-2]


def _bins(n, nbins, kind, seed):
    rng = np.random.default_rng(seed)
    if kind == "uniform":
        return rng.integers(0, nbins, n).astype(np.int32)
    if kind == "sorted":
        return np.sort(rng.integers(0, nbins, n)).astype(np.int32)
    if kind == "one":
        return np.full(n, nbins // 2, np.int32)
    # "outside": a fifth of the entries outside [0, nbins)
    b = rng.integers(0, nbins, n).astype(np.int64)
    bad = rng.random(n) < 0.2
    b[bad] = rng.choice(np.array([-1, -(1 << 31), nbins, nbins + 5, (1 << 31) - 1], np.int64), bad.sum())
    return b.astype(np.int32)


@pytest.mark.parametrize("kind", ["uniform", "sorted", "one", "outside"])
@pytest.mark.parametrize("nbins", NBINS)
@pytest.mark.parametrize("n", SIZES)
def test_histogram_and_offsets(kind, nbins, n):
    bins = _bins(n, nbins, kind, seed=n * 7 + nbins)
    counts = gpu_bins(bins, nbins, False)
    assert np.array_equal(counts, oracle.histogram(bins, nbins)[0])
    offs = gpu_bins(bins, nbins, True)
    assert np.array_equal(offs, oracle.bin_offsets(bins, nbins)[0])


@pytest.mark.parametrize("nbins", [200, 300, 5000, 40000])
def test_unaligned_bins(nbins):
    """Bins not 16-byte aligned (element loads) on the per-warp (<= 1024
    bins), per-CTA (<= 32768) and global-atomic histograms."""
    bins = _bins(100003, nbins, "outside", 1)
    for off in (1, 2, 3):
        assert np.array_equal(gpu_bins(bins, nbins, True, off=off), oracle.bin_offsets(bins, nbins)[0])


def test_csr_rows_workload():
    """The benchmark's COO matrix (2^22 sorted rows, about 2^27 entries) -> CSR row offsets."""
    import torch
    from stream_compaction_gb300 import synth
    spec = synth.WORKLOADS["csr_rows_2^22"]
    rt = synth.make_torch(spec, device="cuda")
    torch.cuda.synchronize()
    rows = rt.cpu().numpy()
    nrows = spec["nrows"]
    offs = gpu_bins(rows, nrows, True)
    assert np.array_equal(offs, oracle.bin_offsets(rows, nrows)[0])
    assert offs[-1] == rows.size


def test_digit_bins_workload():
    import torch
    from stream_compaction_gb300 import synth
    spec = synth.WORKLOADS["digit_bins_n2^27"]
    bt = synth.make_torch(spec, device="cuda")
    torch.cuda.synchronize()
    bins = bt.cpu().numpy()
    assert np.array_equal(gpu_bins(bins, 256, True), oracle.bin_offsets(bins, 256)[0])
