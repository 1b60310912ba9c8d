"""GPU parity: radix sort digit passes and the full 32-bit sort against the CPU
oracle, exactly (a stable pass has exactly one correct output)."""
import numpy as np
import pytest

import oracle
from gpu_helpers import ensure_lib, stream, to_device, to_host

pytestmark = pytest.mark.gpu

SIZES = [1, 2, 100, 4095, 4096, 4097, 3 * 4096 + 5, 100003, (1 << 20) + 17, 3 * (1 << 20) + 77]
DIGITS = [(0, 8), (8, 8), (24, 8), (3, 5), (31, 1), (28, 4)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _keys(n, kind, seed):
    rng = np.random.default_rng(seed)
    k = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
    if kind == "equal":
        k[:] = 0x12345678
    elif kind == "few":
        k = np.array([7, 0xFFFFFFFF, 0x80000000, 256], np.uint32)[rng.integers(0, 4, n)]
    elif kind == "sorted":
        k = np.sort(k)
    elif kind == "reversed":
        k = np.sort(k)[::-1].copy()
    elif kind == "low":
        k &= np.uint32(0x3FF)                       # only two low digits vary
    return k


def gpu_pass(keys, shift, bits, off=0):
    import stream_compaction_gb300 as sc
    n = keys.size
    _, kin = to_device(keys, off)
    _, kout = to_device(np.zeros_like(keys), off)
    st = sc.sc_radix_pass_u32(kin.data_ptr(), kout.data_ptr(), n, shift, bits, stream())
    assert st == sc.SC_OK, sc.status_string(st)
    assert sc.sc_get_device_error(stream()) == sc.SC_OK
    return to_host(kout, keys)


def gpu_sort(keys, off=0, inplace=False):
    import stream_compaction_gb300 as sc
    n = keys.size
    _, kin = to_device(keys, off)
    kout = kin if inplace else to_device(np.zeros_like(keys), off)[1]
    _, tmp = to_device(np.zeros_like(keys))
    st = sc.sc_radix_sort_u32(kin.data_ptr(), kout.data_ptr(), tmp.data_ptr(), n, stream())
    assert st == sc.SC_OK, sc.status_string(st)
    assert sc.sc_get_device_error(stream()) == sc.SC_OK
    return to_host(kout, keys)


def _same(a, b):
    bad = np.flatnonzero(a != b)
    assert bad.size == 0, "%d keys differ, first at %d" % (bad.size, bad[0])


@pytest.mark.parametrize("shift,bits", DIGITS)
@pytest.mark.parametrize("n", SIZES)
def test_radix_pass(shift, bits, n):
    for kind in ("uniform", "few", "equal"):
        k = _keys(n, kind, seed=n + shift * 7 + bits)
        _same(gpu_pass(k, shift, bits), oracle.radix_pass(k, shift, bits))


@pytest.mark.parametrize("kind", ["uniform", "few", "equal", "sorted", "reversed", "low"])
@pytest.mark.parametrize("n", SIZES)
def test_radix_sort(kind, n):
    k = _keys(n, kind, seed=n * 3 + len(kind))
    got = gpu_sort(k)
    _same(got, oracle.radix_sort(k))
    _same(got, np.sort(k))


@pytest.mark.parametrize("variant", range(6))
def test_radix_ranking_variants(variant):
    """Every ranking split (digit bits by match vs by ballots) gives the same stable pass."""
    import stream_compaction_gb300 as sc
    assert sc.sc_set_radix_variant(variant) == sc.SC_OK
    try:
        for n, kind in ((3 * 4096 + 5, "uniform"), (100003, "few"), ((1 << 20) + 17, "uniform")):
            k = _keys(n, kind, seed=variant * 11 + n)
            for shift, bits in ((0, 8), (24, 8), (3, 5), (31, 1)):
                _same(gpu_pass(k, shift, bits), oracle.radix_pass(k, shift, bits))
            _same(gpu_sort(k), np.sort(k))
    finally:
        sc.sc_set_radix_variant(0)


def test_radix_unaligned_and_inplace():
    k = _keys(9 * 4096 + 11, "uniform", 5)
    ref = np.sort(k)
    _same(gpu_sort(k, off=1), ref)
    _same(gpu_sort(k, inplace=True), ref)
    _same(gpu_pass(k, 8, 8, off=3), oracle.radix_pass(k, 8, 8))


def test_radix_argument_checks():
    import stream_compaction_gb300 as sc
    _, a = to_device(np.zeros(64, np.uint32))
    _, b = to_device(np.zeros(64, np.uint32))
    p, q, s = a.data_ptr(), b.data_ptr(), stream()
    assert sc.sc_radix_pass_u32(p, q, 64, 0, 0, s) == sc.SC_ERR_INVALID      # bits
    assert sc.sc_radix_pass_u32(p, q, 64, 0, 9, s) == sc.SC_ERR_INVALID
    assert sc.sc_radix_pass_u32(p, q, 64, 32, 8, s) == sc.SC_ERR_INVALID     # shift
    assert sc.sc_radix_pass_u32(p, p + 16, 64, 0, 8, s) == sc.SC_ERR_INVALID  # overlap
    assert sc.sc_radix_sort_u32(p, q, q, 64, s) == sc.SC_ERR_INVALID          # tmp overlaps out
    assert sc.sc_radix_sort_u32(p, p, q, 64, s) == sc.SC_OK                    # in place


def test_sort_workload_full_size():
    """2^27 full-range keys (the benchmark's workload) against np.sort."""
    import torch
    from stream_compaction_gb300 import synth
    spec = synth.WORKLOADS["uint32_sort_n2^27"]
    kt = synth.make_torch(spec, device="cuda")
    torch.cuda.synchronize()
    k = kt.cpu().numpy().view(np.uint32)
    _same(gpu_sort(k), np.sort(k))
