"""GPU parity: single-pass scans against the CPU oracle, element by element.

Integer sums, int32 max and affine composition must match bit for bit; float32
sums must satisfy |y_gpu[i] - y_ref[i]| <= 1e-5 * sum_{k<=i} |x[k]| (fp64
oracle).  Sizes span one element to many tiles with ragged tails; pointers are
16-byte aligned (vector path) and merely element-aligned (scalar path); scans
also run in place.
"""
import numpy as np
import pytest

import oracle
from gpu_helpers import check_f32, ensure_lib, gpu_scan
from stream_compaction_gb300 import synth

pytestmark = pytest.mark.gpu

T = 4096  # default tile of the 4-byte operators (affine: 2048)
SIZES = [1, 2, 3, 31, 32, 33, 1000, T - 1, T, T + 1, 2 * T - 1, 2 * T + 1, 2 * T + 2, 4 * T - 1, 4 * T + 1,
         7 * T + 13, 33 * T + 5, (1 << 20) + 17, 100 * T + 4095, 1000 * T + 17, 3000 * T - 1]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _input(kind, n, seed):
    rng = np.random.default_rng(seed)
    if kind == "i32":
        return rng.integers(-1000, 1000, n).astype(np.int32)
    if kind == "u32":
        return rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
    if kind == "maxi32":
        return rng.integers(-(1 << 31), (1 << 31) - 1, n, endpoint=True).astype(np.int32)
    if kind == "f32":
        return rng.uniform(-1, 1, n).astype(np.float32)
    if kind == "affine":
        return rng.integers(0, 1 << 32, (n, 2), dtype=np.uint64).astype(np.uint32)
    raise ValueError(kind)


CASES = [("i32", "sum"), ("u32", "sum"), ("maxi32", "max"), ("affine", "affine"), ("f32", "sum")]


@pytest.mark.parametrize("kind,op", CASES)
@pytest.mark.parametrize("exclusive", [False, True])
@pytest.mark.parametrize("n", SIZES)
def test_scan_sizes(kind, op, exclusive, n):
    x = _input(kind, n, seed=n * 7 + len(kind))
    y = gpu_scan(x, op, exclusive)
    ref = oracle.scan(x, op, exclusive)
    if kind == "f32":
        check_f32(y, ref, oracle.abs_prefix(x), "n=%d" % n)
    else:
        assert np.array_equal(y, ref)


@pytest.mark.parametrize("kind,op", CASES)
@pytest.mark.parametrize("exclusive", [False, True])
@pytest.mark.parametrize("n", [T + 3, 5 * T, 9 * T + 1])
def test_scan_unaligned_and_inplace(kind, op, exclusive, n):
    x = _input(kind, n, seed=99 + n)
    ref = oracle.scan(x, op, exclusive)
    off = 2 if kind == "affine" else 1  # element-aligned, not 16-byte aligned
    for y in (gpu_scan(x, op, exclusive, offset=off), gpu_scan(x, op, exclusive, inplace=True),
              gpu_scan(x, op, exclusive, offset=off, inplace=True)):
        if kind == "f32":
            check_f32(y, ref, oracle.abs_prefix(x))
        else:
            assert np.array_equal(y, ref)


def test_closed_forms_on_gpu():
    n = 3 * T + 11
    ones = np.ones(n, dtype=np.uint32)
    assert np.array_equal(gpu_scan(ones, "sum", True), np.arange(n, dtype=np.uint32))
    allf = np.full(n, 0xFFFFFFFF, dtype=np.uint32)
    assert np.array_equal(gpu_scan(allf, "sum", False),
                          (-(np.arange(n, dtype=np.int64) + 1)).astype(np.int32).view(np.uint32))
    # float32 all ones: exact integers below 2^24
    fo = np.ones(n, dtype=np.float32)
    assert np.array_equal(gpu_scan(fo, "sum", True), np.arange(n, dtype=np.float32))
    # identities in front of exclusive scans
    assert gpu_scan(np.array([5, 6], np.int32), "max", True)[0] == np.iinfo(np.int32).min
    ya = gpu_scan(np.array([[3, 4], [5, 6]], np.uint32), "affine", True)
    assert ya[0].tolist() == [1, 0]


def _num_variants():
    import stream_compaction_gb300 as sc
    v = 0
    while sc.sc_scan_variant_info(v)[0] == sc.SC_OK:
        v += 1
    return v


@pytest.mark.parametrize("variant", range(30))
def test_uint32_variants(variant):
    import stream_compaction_gb300 as sc
    if variant >= _num_variants():
        pytest.skip("variant not compiled")
    assert sc.sc_set_scan_variant(variant) == sc.SC_OK
    try:
        for n in (1, 4097, 8191, 8192, 8193, 16385, 77 * 4096 + 1234, 301 * 8192 + 77):
            x = _input("u32", n, seed=variant * 1000 + n)
            for ex in (False, True):
                assert np.array_equal(gpu_scan(x, "sum", ex), oracle.scan(x, "sum", ex)), (variant, n, ex)
                assert np.array_equal(gpu_scan(x, "sum", ex, offset=1), oracle.scan(x, "sum", ex))
        # segmented scans take the variant's shape where it has a segmented form
        from test_gpu_segmented import _heads, gpu_segmented
        n = 77 * 4096 + 1234
        x = _input("u32", n, seed=variant + 5)
        for density in (1e-4, 3e-3):
            h = _heads(n, density, seed=variant)
            for ex in (False, True):
                got = gpu_segmented(x, h, "sum", ex)
                assert np.array_equal(got, oracle.scan_segmented(x, h, "sum", ex)), (variant, density, ex)
    finally:
        sc.sc_set_scan_variant(0)


def test_repeated_runs_are_exact():
    """A passing run proves little for a racy protocol: repeat with many grid sizes."""
    import stream_compaction_gb300 as sc
    rng = np.random.default_rng(5)
    for it in range(60):
        sc.sc_set_scan_variant(it % _num_variants())
        n = int(rng.integers(1, 3 << 20))
        x = _input("u32", n, seed=it)
        assert np.array_equal(gpu_scan(x, "sum", it % 2 == 0), oracle.scan(x, "sum", it % 2 == 0)), (it, n)
    sc.sc_set_scan_variant(0)


# ------------------------------------------------------- benchmark workloads
def _workload(name):
    import torch
    spec = synth.WORKLOADS[name]
    xt = synth.make_torch(spec, device="cuda")
    torch.cuda.synchronize()
    x = xt.cpu().numpy()
    return x


def test_workload_int32_sum_n1048593():
    x = _workload("int32_sum_n1048593")
    for ex in (False, True):
        assert np.array_equal(gpu_scan(x, "sum", ex), oracle.scan(x, "sum", ex))


def test_workload_float32_exsum_n2p26():
    x = _workload("float32_exsum_n2^26")
    y = gpu_scan(x, "sum", True)
    worst = check_f32(y, oracle.scan(x, "sum", True), oracle.abs_prefix(x), "float32 n=2^26")
    assert worst < 1e-5


def test_workload_int32_max_n2p27():
    x = _workload("int32_max_n2^27").view(np.int32)
    assert np.array_equal(gpu_scan(x, "max", False), oracle.scan(x, "max", False))


def test_workload_affine_n2p26():
    x = _workload("affine_u32_n2^26").view(np.uint32)
    assert np.array_equal(gpu_scan(x, "affine", False), oracle.scan(x, "affine", False))


def test_workload_uint32_exsum_n2p30():
    """The headline workload at full size: every one of the 2^30 outputs is compared."""
    x = _workload("uint32_exsum_n2^30").view(np.uint32)
    y = gpu_scan(x, "sum", True)
    ref = oracle.scan(x, "sum", True)
    assert np.array_equal(y, ref)


def test_float32_sum_infinities_cross_tiles():
    """Infinities and NaN carried between tiles and chunks stay what a float32 sum
    makes of them: +inf after a +inf, NaN once -inf has followed, in the
    persistent scan and in the persistent segmented scan (a head resets)."""
    from test_gpu_segmented import gpu_segmented
    n = (1 << 22) + 3 * 8192 + 5                      # persistent kernels: several tiles and chunks
    rng = np.random.default_rng(17)
    x = rng.uniform(-1, 1, n).astype(np.float32)
    x[5000] = np.inf
    x[(1 << 20) + 77] = -np.inf
    ax = np.abs(x.astype(np.float64))
    scale = np.cumsum(ax)                                # the float32 bound's scale (inf past an infinity)
    for ex in (False, True):
        y = gpu_scan(x, "sum", ex)
        ref = oracle.scan(x, "sum", ex)
        assert np.array_equal(np.isnan(y), np.isnan(ref)) and np.array_equal(np.isposinf(y), np.isposinf(ref))
        fin = np.isfinite(ref)
        assert np.all(np.abs(y[fin] - ref[fin]) <= 1e-5 * scale[fin])
    h = np.zeros(n, np.uint8)
    h[[100000, 1 << 20, (1 << 20) + 500000]] = 1          # the second -inf segment ends at the third head
    starts = [0, 100000, 1 << 20, (1 << 20) + 500000, n]
    seg_scale = np.concatenate([np.cumsum(ax[a:b]) for a, b in zip(starts[:-1], starts[1:])])  # restarts at each head
    for ex in (False, True):
        y = gpu_segmented(x, h, "sum", ex)
        ref = oracle.scan_segmented(x, h, "sum", ex)
        assert np.array_equal(np.isnan(y), np.isnan(ref)) and np.array_equal(np.isinf(y), np.isinf(ref))
        fin = np.isfinite(ref)
        assert np.all(np.abs(y[fin] - ref[fin]) <= 1e-5 * seg_scale[fin])


# ------------------------------------- persistent scan: in place, boundaries
# Sizes just past the short-scan limit (2^22) and around the persistent
# kernel's 8192-element tiles and 2-tile chunks, each with a ragged end.
P_SIZES = [(1 << 22) + 1, (1 << 22) + 8192, (1 << 23) - 1, (1 << 22) + 16384 + 1, 3 * (1 << 22) + 77]
P_KINDS = [("u32", "sum"), ("f32", "sum"), ("maxi32", "max"), ("affine", "affine"), ("i64", "sum"),
           ("f64", "sum"), ("maxcount", "maxcount")]


def _p_input(kind, op, n, seed):
    if kind in ("i64", "f64", "maxcount"):
        from test_gpu_ops import make_input
        return make_input(kind, op, n, seed)
    return _input(kind, n, seed)


@pytest.mark.parametrize("kind,op", P_KINDS)
@pytest.mark.parametrize("n", P_SIZES)
def test_persistent_scan_in_place_at_boundaries(kind, op, n):
    """16-byte aligned arrays above the short-scan limit take the persistent
    kernel, whose pass 2 re-reads each tile from global memory while the TMA
    stores of other tiles are in flight: in place and out of place, inclusive
    and exclusive, every output against the oracle."""
    import stream_compaction_gb300 as sc
    from gpu_helpers import check_f64
    x = _p_input(kind, op, n, seed=n % 1000 + len(kind))
    for exclusive in (False, True):
        ref = oracle.scan(x, op, exclusive)
        for inplace in (False, True):
            y = gpu_scan(x, op, exclusive, inplace=inplace)
            assert sc.sc_debug_last_path() == sc.SC_PATH_SCAN_PERSISTENT, (kind, n)
            what = "%s n=%d excl=%d inplace=%d" % (kind, n, exclusive, inplace)
            if kind == "f32":
                check_f32(y, ref, oracle.abs_prefix(x), what)
            elif kind == "f64":
                check_f64(y, ref, oracle.abs_prefix(x), what)
            else:
                assert np.array_equal(y, ref), what


@pytest.mark.parametrize("kind,op", [("affine", "affine"), ("i64", "sum"), ("f64", "sum"), ("maxcount", "maxcount")])
@pytest.mark.parametrize("n", [1 << 20, (1 << 20) + 1, (1 << 20) + 2 * 4096 + 3, (1 << 21) + 77])
def test_eight_byte_short_scan_limit(kind, op, n):
    """8-byte elements take the one-tile-per-CTA kernel up to 2^20 elements and
    the persistent kernel above (their crossover measured on GB300); both
    sides of the limit, in place and not, against the oracle."""
    import stream_compaction_gb300 as sc
    from gpu_helpers import check_f64
    x = _p_input(kind, op, n, seed=n % 991 + len(kind))
    want = sc.SC_PATH_SCAN_ONE_TILE if n <= (1 << 20) else sc.SC_PATH_SCAN_PERSISTENT
    for exclusive in (False, True):
        ref = oracle.scan(x, op, exclusive)
        for inplace in (False, True):
            y = gpu_scan(x, op, exclusive, inplace=inplace)
            assert sc.sc_debug_last_path() == want, (kind, n)
            what = "%s n=%d excl=%d inplace=%d" % (kind, n, exclusive, inplace)
            if kind == "f64":
                check_f64(y, ref, oracle.abs_prefix(x), what)
            else:
                assert np.array_equal(y, ref), what


@pytest.mark.parametrize("kind,op,n", [("u32", "sum", (1 << 24) + 4097), ("affine", "affine", (1 << 23) + 5),
                                       ("f32", "sum", (1 << 24) + 3)])
def test_host_scan_in_place_across_chunks(kind, op, n):
    """sc_scan_host with h_in == h_out: the staging chunks are 64 MiB (2^24
    four-byte or 2^23 eight-byte elements), so these sizes carry the running
    total across a chunk boundary into a ragged last chunk."""
    import stream_compaction_gb300 as sc
    from gpu_helpers import CODE, OPC, stream
    x = _input(kind, n, seed=n % 977)
    for exclusive in (False, True):
        h = np.ascontiguousarray(x.copy())
        code = CODE["affine" if kind == "affine" else kind]
        st = sc.sc_scan_host(code, OPC[op], int(exclusive), h.ctypes.data, h.ctypes.data, n, stream())
        assert st == sc.SC_OK, sc.status_string(st)
        ref = oracle.scan(x, op, exclusive)
        if kind == "f32":
            check_f32(h, ref, oracle.abs_prefix(x), "host in place")
        else:
            assert np.array_equal(h, ref)


def test_float32_statuses_across_epoch_wraps_and_workspace_reuse():
    """Float32 sums carry float-float pairs in one-word look-back statuses with
    a 7-bit epoch, so the library clears the status area whenever a stream's
    epoch would pass 127.  Many calls on one stream, float32 sums interleaved
    with uint32 sums (which keep counting epochs past 127), the hierarchical
    variant and a radix pass (both leave other data where statuses go), each
    checked against the oracle."""
    import stream_compaction_gb300 as sc
    from gpu_helpers import stream
    rng = np.random.default_rng(11)
    xs = {n: rng.uniform(-1, 1, n).astype(np.float32) for n in (100003, (1 << 22) + 8195)}
    refs = {n: oracle.scan(x, "sum", True) for n, x in xs.items()}
    scales = {n: oracle.abs_prefix(x) for n, x in xs.items()}
    u = _input("u32", 300007, seed=5)
    uref = oracle.scan(u, "sum", False)
    keys = _input("u32", 70001, seed=6)
    for it in range(420):
        n = (1 << 22) + 8195 if it % 7 == 3 else 100003
        y = gpu_scan(xs[n], "sum", True)
        check_f32(y, refs[n], scales[n], "it %d" % it)
        if it % 3 == 0:
            assert np.array_equal(gpu_scan(u, "sum", False), uref)
        if it % 50 == 7:
            assert np.array_equal(gpu_scan(u, "sum", False, hierarchical=True), uref)
        if it % 50 == 19:
            import torch
            kd = torch.from_numpy(keys.view(np.int32)).cuda()
            ko = torch.empty_like(kd)
            assert sc.sc_radix_pass_u32(kd.data_ptr(), ko.data_ptr(), keys.size, 8, 8, stream()) == sc.SC_OK
            assert np.array_equal(ko.cpu().numpy().view(np.uint32), oracle.radix_pass(keys, 8, 8))
