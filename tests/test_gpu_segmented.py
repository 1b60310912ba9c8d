"""GPU parity: segmented scans with head flags against the CPU oracle.

Head densities from none to every element, ragged tiles of both element
sizes, one or many tiles, flags and data that are not 16-byte aligned,
in-place scans, every operator family; plus the pages' use of a segmented max
scan (the first element of each segment that satisfies a predicate).
"""
import numpy as np
import pytest

import oracle
from gpu_helpers import CODE, OPC, check_f32, check_f64, ensure_lib, kind_of, same_float, stream, to_device, to_host
from test_gpu_ops import make_input

pytestmark = pytest.mark.gpu

CASES = [("i32", "sum"), ("u32", "sum"), ("i32", "max"), ("f32", "sum"), ("affine", "affine"), ("u32", "xor"),
         ("i32", "min"), ("u32", "prod"), ("i64", "sum"), ("u64", "and"), ("i64", "max"), ("f32", "max"),
         ("f64", "sum"), ("f64", "min"), ("maxcount", "maxcount")]
SIZES = [1, 33, 2047, 4097, 3 * 4096 + 5, 100003, (1 << 20) + 17, 3 * (1 << 21) + 77]
DENSITIES = [0.0, 1e-4, 0.01, 0.3, 1.0]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _input(kind, op, n, seed):
    if kind == "affine":
        rng = np.random.default_rng(seed)
        return rng.integers(0, 1 << 32, (n, 2), dtype=np.uint64).astype(np.uint32)
    return make_input(kind, op, n, seed)


def _heads(n, density, seed):
    rng = np.random.default_rng(seed)
    return (rng.random(n) < density).astype(np.uint8)


def gpu_segmented(x, heads, op, exclusive, offset=0, hoff=0, inplace=False):
    import torch
    import stream_compaction_gb300 as sc
    n = x.shape[0]
    _, xin = to_device(x, offset)
    xout = xin if inplace else to_device(np.zeros_like(x), offset)[1]
    hbase = torch.zeros(n + hoff + 16, dtype=torch.uint8, device="cuda")
    hv = hbase[hoff:hoff + n]
    hv.copy_(torch.from_numpy(heads))
    k = kind_of(x, op)
    st = sc.sc_scan_segmented(CODE[k], OPC[op], int(exclusive), xin.data_ptr(), hv.data_ptr(), xout.data_ptr(), n,
                              stream())
    assert st == sc.SC_OK, sc.status_string(st)
    assert sc.sc_get_device_error(stream()) == sc.SC_OK
    return to_host(xout, x)


def _check(kind, op, x, heads, y, ref):
    if kind == "f32" and op == "sum":
        s = np.abs(x.astype(np.float64))
        # the bound's scale restarts at each head, like the scan
        scale = oracle.scan_segmented(s, heads, "sum", False)
        check_f32(y, ref, scale)
    elif kind == "f64" and op == "sum":
        check_f64(y, ref, oracle.scan_segmented(np.abs(x), heads, "sum", False))
    elif kind in ("f32", "f64"):
        assert same_float(y, ref)
    else:
        assert np.array_equal(y, ref)


@pytest.mark.parametrize("kind,op", CASES)
@pytest.mark.parametrize("density", DENSITIES)
@pytest.mark.parametrize("n", SIZES)
def test_segmented(kind, op, density, n):
    x = _input(kind, op, n, seed=n + int(density * 1000))
    h = _heads(n, density, seed=n * 3 + 1)
    for ex in (False, True):
        y = gpu_segmented(x, h, op, ex)
        _check(kind, op, x, h, y, oracle.scan_segmented(x, h, op, ex))


@pytest.mark.parametrize("kind,op", CASES)
def test_segmented_unaligned_and_inplace(kind, op):
    n = 9 * 4096 + 11
    x = _input(kind, op, n, seed=5)
    h = _heads(n, 0.002, seed=6)
    off = 2 if kind in ("affine", "maxcount") else 1
    for ex in (False, True):
        ref = oracle.scan_segmented(x, h, op, ex)
        for kw in (dict(offset=off), dict(hoff=3), dict(inplace=True), dict(offset=off, hoff=1, inplace=True)):
            _check(kind, op, x, h, gpu_segmented(x, h, op, ex, **kw), ref)


def test_segmented_heads_on_tile_boundaries():
    """Heads exactly at tile starts, just before and just after them."""
    n = 40 * 4096 + 5
    x = make_input("u32", "xor", n, seed=9)
    for pos in ([4096 * k for k in range(1, 40)], [4096 * k - 1 for k in range(1, 40)],
                [4096 * k + 1 for k in range(1, 40)], [2048 * k for k in range(1, 80)]):
        h = np.zeros(n, np.uint8)
        h[pos] = 1
        for ex in (False, True):
            assert np.array_equal(gpu_segmented(x, h, "xor", ex), oracle.scan_segmented(x, h, "xor", ex))
        xs = make_input("i64", "sum", n, seed=10)
        assert np.array_equal(gpu_segmented(xs, h, "sum", True), oracle.scan_segmented(xs, h, "sum", True))


def test_first_satisfying_element_per_segment():
    """A segmented exclusive max scan of the predicate: the first element of each
    segment that satisfies it is where it holds and nothing before it (in the
    segment) did."""
    rng = np.random.default_rng(12)
    n = (1 << 20) + 333
    p = (rng.random(n) < 0.05).astype(np.int32)
    h = _heads(n, 0.001, seed=13)
    seen = gpu_segmented(p, h, "max", True)
    first = (p == 1) & (seen <= 0)
    ref = oracle.scan_segmented(p, h, "max", True)
    assert np.array_equal(seen, ref)
    starts = np.flatnonzero(np.concatenate([[1], h[1:]]))
    want = np.zeros(n, bool)
    for a, b in zip(starts, list(starts[1:]) + [n]):
        hit = np.flatnonzero(p[a:b])
        if hit.size:
            want[a + hit[0]] = True
    assert np.array_equal(first, want)


def test_segmented_equals_batched_rows():
    import stream_compaction_gb300 as sc
    from gpu_helpers import gpu_batched
    rows, cols = 300, 5000
    x = make_input("i32", "min", rows * cols, seed=3)
    h = np.zeros(rows * cols, np.uint8)
    h[::cols] = 1
    for ex in (False, True):
        assert np.array_equal(gpu_segmented(x, h, "min", ex), gpu_batched(x.reshape(rows, cols), "min", ex).ravel())


def test_segmented_workload_full_size():
    """The benchmark's segmented-sum workload at full size, against the oracle."""
    import torch
    from stream_compaction_gb300 import synth
    spec = synth.WORKLOADS["int32_segsum_n2^27"]
    xt = synth.make_torch(spec, device="cuda")
    torch.cuda.synchronize()
    x = xt.cpu().numpy()
    h = synth.make_heads_np(spec)
    assert np.array_equal(gpu_segmented(x, h, "sum", True), oracle.scan_segmented(x, h, "sum", True))
    spec = synth.WORKLOADS["float32_segsum_n2^27"]
    xt = synth.make_torch(spec, device="cuda")
    torch.cuda.synchronize()
    x = xt.cpu().numpy()
    scale = oracle.scan_segmented(np.abs(x.astype(np.float64)), h, "sum", False)
    check_f32(gpu_segmented(x, h, "sum", True), oracle.scan_segmented(x, h, "sum", True), scale)


@pytest.mark.parametrize("op", ["sum", "max"])
def test_segmented_persistent_tile_and_chunk_boundaries(op):
    """int32 sums and max segmented by heads run on the persistent kernel
    (8192-element tiles, 2-tile chunks, flags bulk-copied with each tile):
    heads on, just before and just after tile and chunk starts, a head only
    in the ragged last tile, heads everywhere, and sizes around tile
    multiples; the one-tile-per-CTA kernel (scan variant 1) must agree."""
    import stream_compaction_gb300 as sc
    T, CH = 8192, 16384
    for n in (T, T + 1, 2 * CH - 1, 2 * CH, 7 * CH + T + 3, 64 * CH + 5):
        x = make_input("i32", op, n, seed=n)
        cases = [np.zeros(n, np.uint8), np.ones(n, np.uint8)]
        for stride, shift in ((T, 0), (T, -1), (T, 1), (CH, 0), (CH, -1), (CH, 1)):
            h = np.zeros(n, np.uint8)
            idx = np.arange(stride + shift, n, stride)
            h[idx[(idx >= 0) & (idx < n)]] = 1
            cases.append(h)
        h = np.zeros(n, np.uint8)
        h[n - 1] = 7                                   # any nonzero byte is a head
        cases.append(h)
        for h in cases:
            for ex in (False, True):
                ref = oracle.scan_segmented(x, h, op, ex)
                got = gpu_segmented(x, h, op, ex)
                assert np.array_equal(got, ref), (n, op, ex)
        assert sc.sc_set_scan_variant(1) == sc.SC_OK
        try:
            assert np.array_equal(gpu_segmented(x, cases[-2], op, True), oracle.scan_segmented(x, cases[-2], op, True))
        finally:
            sc.sc_set_scan_variant(0)
