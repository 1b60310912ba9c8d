"""GPU parity: batched row scans, fused compaction, the hierarchical comparison
variant and the host-buffer pipeline, each against the CPU oracle."""
import math

import numpy as np
import pytest

import oracle
from gpu_helpers import check_f32, ensure_lib, gpu_batched, gpu_compact, gpu_scan, stream, to_device
from stream_compaction_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


# ------------------------------------------------------------- batched rows
SHAPES = [(1, 1), (1, 5000), (3, 1), (7, 3), (100, 17), (5, 4096), (3, 4097), (2, 10000), (1000, 33),
          (64, 8195), (257, 4095), (9, 12289), (4096, 16), (20000, 33), (300, 1000), (50, 2047), (8192, 64),
          (2048, 256)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("exclusive", [False, True])
@pytest.mark.parametrize("kind", ["i32", "max", "f32", "affine"])
def test_batched(shape, exclusive, kind):
    rows, cols = shape
    rng = np.random.default_rng(rows * 31 + cols)
    if kind == "i32":
        x, op = rng.integers(0, 256, shape).astype(np.int32), "sum"
    elif kind == "max":
        x, op = rng.integers(-(1 << 31), (1 << 31) - 1, shape, endpoint=True).astype(np.int32), "max"
    elif kind == "f32":
        x, op = rng.uniform(-1, 1, shape).astype(np.float32), "sum"
    else:
        x, op = rng.integers(0, 1 << 32, (rows, cols, 2), dtype=np.uint64).astype(np.uint32), "affine"
    y = gpu_batched(x, op, exclusive)
    ref = oracle.scan_batched(x, op, exclusive)
    if kind == "f32":
        s = np.stack([oracle.abs_prefix(r) for r in x])
        check_f32(y.reshape(-1), ref.reshape(-1), s.reshape(-1))
    else:
        assert np.array_equal(y, ref)


@pytest.mark.parametrize("kind,op", [("i32", "sum"), ("u32", "xor"), ("i32", "min"), ("u32", "prod"), ("f32", "max"),
                                     ("f32", "sum"), ("i32", "max")])
@pytest.mark.parametrize("shape", [(8192, 1), (8192, 5), (4099, 3), (1000, 33), (300, 1000), (20, 8191), (9, 12289),
                                   (3, 40000), (1024, 64), (64, 4096), (7, 8192), (3000, 32), (70000, 2), (513, 16),
                                   (40000, 33), (3000, 1000), (700, 2047), (200, 8191), (300000, 7)])
def test_batched_rows_persistent(kind, op, shape):
    """Rows of 4-byte elements on 16-byte aligned arrays of at least one tile:
    on the persistent rows kernel (sum, int32 max, float32 sum) lengths that
    divide 8192 (every tile whole rows) and, out of place, other lengths up to
    8192 (a CTA carries the open row from tile to tile and reads back the part
    before its first tile: the shapes of 1.3M-3M elements give CTAs several
    tiles); other operators on the one-tile kernel when the length divides
    4096; the rest on the persistent segmented kernel with heads at the
    multiples of the row length.  Rows shorter than, equal to and longer than
    a thread's 32 items, a warp's part and the 8192-element tile, with ragged
    last tiles, in place and not."""
    import stream_compaction_gb300 as sc
    from gpu_helpers import CODE, OPC, dev_buffer, stream, to_host
    from test_gpu_ops import make_input
    rows, cols = shape
    x = make_input(kind, op, rows * cols, seed=rows + cols).reshape(rows, cols)
    for exclusive in (False, True):
        ref = oracle.scan_batched(x, op, exclusive)
        for inplace in (False, True):
            _, xin = to_device(x)
            xout = xin if inplace else dev_buffer(xin.numel(), xin.dtype)[1]
            st = sc.sc_scan_batched(CODE[kind], OPC[op], int(exclusive), xin.data_ptr(), xout.data_ptr(), rows, cols,
                                    stream())
            assert st == sc.SC_OK, sc.status_string(st)
            rows_op = (kind, op) in (("i32", "sum"), ("u32", "sum"), ("f32", "sum"), ("i32", "max"))
            # rows dividing 8192 always; other lengths up to 8192 when out != in
            rows_kernel = rows_op and (8192 % cols == 0 or (cols <= 8192 and not inplace))
            want = (sc.SC_PATH_ROWS_PERSISTENT if rows_kernel else
                    sc.SC_PATH_SCAN_ONE_TILE if 4096 % cols == 0 else sc.SC_PATH_SEGSCAN_PERSISTENT)
            assert sc.sc_debug_last_path() == want, shape
            assert sc.sc_get_device_error(stream()) == sc.SC_OK
            y = to_host(xout, x)
            if kind == "f32" and op == "sum":
                s_abs = np.stack([oracle.abs_prefix(r) for r in x])
                check_f32(y.reshape(-1), ref.reshape(-1), s_abs.reshape(-1))
            elif kind == "f32":
                from gpu_helpers import same_float
                assert same_float(y, ref), (shape, exclusive, inplace)
            else:
                assert np.array_equal(y, ref), (shape, exclusive, inplace)


def test_workload_int32_rows_65536x4096():
    import torch
    spec = synth.WORKLOADS["int32_rows_65536x4096"]
    xt = synth.make_torch(spec, device="cuda")
    torch.cuda.synchronize()
    x = xt.cpu().numpy().reshape(65536, 4096)
    y = gpu_batched(x, "sum", True)
    assert np.array_equal(y, oracle.scan_batched(x, "sum", True))


@pytest.mark.parametrize("cols", [33, 1000, 2047])
def test_workload_int32_ragged_rows_full_size(cols):
    """The benchmark's ragged-row shapes: the 65536 x 4096 input's first
    rows * cols elements viewed as rows of 33, 1000 and 2047 (tiles start
    inside rows, so every CTA carries the open row from tile to tile and reads
    back the part of its first tile's row before it), on the rows kernel."""
    import torch
    import stream_compaction_gb300 as sc
    spec = synth.WORKLOADS["int32_rows_65536x4096"]
    xt = synth.make_torch(spec, device="cuda")
    rows = xt.numel() // cols
    xt = xt[:rows * cols].contiguous()
    yt = torch.empty_like(xt)
    st = sc.sc_scan_batched(sc.SC_I32, sc.SC_SUM, 1, xt.data_ptr(), yt.data_ptr(), rows, cols, stream())
    assert st == sc.SC_OK, sc.status_string(st)
    assert sc.sc_debug_last_path() == sc.SC_PATH_ROWS_PERSISTENT
    assert sc.sc_get_device_error(stream()) == sc.SC_OK
    x = xt.cpu().numpy().reshape(rows, cols)
    assert np.array_equal(yt.cpu().numpy().reshape(rows, cols), oracle.scan_batched(x, "sum", True))


# ------------------------------------------------------------- compaction
CSIZES = [1, 2, 33, 4095, 4096, 4097, 3 * 4096 + 17, 100003, (1 << 20) + 17]


@pytest.mark.parametrize("n", CSIZES)
@pytest.mark.parametrize("dtype", ["i32", "u32", "f32"])
def test_compact_sizes(n, dtype):
    rng = np.random.default_rng(n)
    if dtype == "i32":
        x = rng.integers(-(1 << 20), 1 << 20, n).astype(np.int32)
    elif dtype == "u32":
        x = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
    else:
        x = rng.uniform(-1, 1, n).astype(np.float32)
    thr = 0 if dtype != "u32" else float(1 << 31)
    for pred in ("gt", "ge", "lt", "le", "eq", "ne"):
        for off in (0, 1):
            out, c, full = gpu_compact(x, pred, thr, offset=off)
            ref, rc = oracle.compact(x, pred, thr)
            assert c == rc and np.array_equal(out, ref), (pred, off)
            if c < n:  # the library never writes past the count
                assert np.all(full[c:n].view(np.int32) == -7)


THRESHOLDS = [0, 0.5, -0.5, -0.0, 1e-45, 3.0, -3.0, 2 ** 31, -2 ** 31, 2 ** 31 - 0.5, 2 ** 32, 2 ** 40,
              -1e300, 1e300, math.inf, -math.inf, math.nan, 0.1, 16777217.0]


@pytest.mark.parametrize("dtype", ["i32", "u32", "f32"])
def test_compact_threshold_canonicalisation(dtype):
    """The kernel compares in the element type; the oracle compares in double.
    Both must agree for thresholds between representable values, out of range,
    infinite and NaN."""
    special = {
        "i32": np.array([0, 1, -1, 2, -2, 3, -3, 2 ** 31 - 1, -2 ** 31, 5, 100, -100], dtype=np.int64).astype(np.int32),
        "u32": np.array([0, 1, 2, 3, 2 ** 31, 2 ** 31 - 1, 2 ** 32 - 1, 5, 100], dtype=np.uint64).astype(np.uint32),
        "f32": np.array([0.0, -0.0, 0.5, -0.5, 0.1, 1e-45, -1e-45, 3.0, 16777216.0, 16777218.0, np.inf, -np.inf,
                         np.nan, 3.4e38, -3.4e38, 2.0 ** 31, 2.0 ** 32, 1.0000001], dtype=np.float32),
    }[dtype]
    x = np.tile(special, 700)
    for thr in THRESHOLDS:
        for pred in ("gt", "ge", "lt", "le", "eq", "ne"):
            out, c, _ = gpu_compact(x, pred, thr)
            ref, rc = oracle.compact(x, pred, thr)
            assert c == rc, (dtype, pred, thr)
            assert np.array_equal(out.view(np.int32), ref.view(np.int32)), (dtype, pred, thr)


def test_compact_all_and_none():
    n = 5 * 4096 + 3
    x = np.arange(1, n + 1, dtype=np.int32)
    out, c, _ = gpu_compact(x, "gt", 0)
    assert c == n and np.array_equal(out, x)
    out, c, _ = gpu_compact(x, "lt", 0)
    assert c == 0


def test_compact_empty():
    import torch
    import stream_compaction_gb300 as sc
    cnt = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    assert sc.sc_compact_if(sc.SC_I32, 0, 0, cnt.data_ptr(), 0, sc.SC_GT, 0.0, stream()) == sc.SC_OK
    assert int(cnt.item()) == 0


def test_workload_int32_compact_gt0_n2p27():
    import torch
    spec = synth.WORKLOADS["int32_compact_gt0_n2^27"]
    xt = synth.make_torch(spec, device="cuda")
    torch.cuda.synchronize()
    x = xt.cpu().numpy()
    out, c, _ = gpu_compact(x, "gt", 0)
    ref, rc = oracle.compact(x, "gt", 0)
    assert c == rc and np.array_equal(out, ref)
    assert abs(c / x.size - 0.5) < 0.01


# ---------------------------------------------------- hierarchical variant
@pytest.mark.parametrize("n", [1, 4095, 4096, 4097, 3 * 4096 + 1, 4096 * 4096 + 17, (1 << 20) + 17])
@pytest.mark.parametrize("kind,op", [("u32", "sum"), ("max", "max"), ("f32", "sum"), ("affine", "affine")])
@pytest.mark.parametrize("exclusive", [False, True])
def test_hierarchical(n, kind, op, exclusive):
    rng = np.random.default_rng(n + 3)
    if kind == "u32":
        x = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
    elif kind == "max":
        x = rng.integers(-(1 << 31), (1 << 31) - 1, n, endpoint=True).astype(np.int32)
    elif kind == "f32":
        x = rng.uniform(-1, 1, n).astype(np.float32)
    else:
        x = rng.integers(0, 1 << 32, (n, 2), dtype=np.uint64).astype(np.uint32)
    y = gpu_scan(x, op, exclusive, hierarchical=True)
    ref = oracle.scan(x, op, exclusive)
    if kind == "f32":
        check_f32(y, ref, oracle.abs_prefix(x))
    else:
        assert np.array_equal(y, ref)


# ---------------------------------------------------- host-buffer pipeline
@pytest.mark.parametrize("n", [1, 5, (1 << 24) - 1, (1 << 24) + 5, 3 * (1 << 24) + 7])
def test_scan_host_u32(n):
    import torch
    import stream_compaction_gb300 as sc
    x = synth.full_u32_np(n, seed=11)
    xt = torch.from_numpy(x.view(np.int32)).pin_memory()
    yt = torch.empty_like(xt).pin_memory()
    for ex in (True, False):
        st = sc.sc_scan_host(sc.SC_U32, sc.SC_SUM, int(ex), xt.data_ptr(), yt.data_ptr(), n, stream())
        assert st == sc.SC_OK
        assert np.array_equal(yt.numpy().view(np.uint32), oracle.scan(x, "sum", ex))


@pytest.mark.parametrize("kind,op", [("f32", "sum"), ("affine", "affine"), ("max", "max")])
def test_scan_host_other_ops(kind, op):
    import torch
    import stream_compaction_gb300 as sc
    n = (1 << 24) + 4099 if kind != "affine" else (1 << 23) + 4099
    rng = np.random.default_rng(1)
    if kind == "f32":
        x = rng.uniform(-1, 1, n).astype(np.float32)
        code = sc.SC_F32
    elif kind == "max":
        x = rng.integers(-(1 << 31), (1 << 31) - 1, n, endpoint=True).astype(np.int32)
        code = sc.SC_I32
    else:
        x = rng.integers(0, 1 << 32, (n, 2), dtype=np.uint64).astype(np.uint32)
        code = sc.SC_AFFINE_U32
    xt = torch.from_numpy(x.view(np.float32) if kind == "f32" else x.view(np.int32)).pin_memory()
    yt = torch.empty_like(xt)  # pageable output also works
    opc = {"sum": sc.SC_SUM, "max": sc.SC_MAX, "affine": sc.SC_COMPOSE}[op]
    st = sc.sc_scan_host(code, opc, 1, xt.data_ptr(), yt.data_ptr(), n, stream())
    assert st == sc.SC_OK
    y = yt.numpy().view(x.dtype).reshape(x.shape)
    ref = oracle.scan(x, op, True)
    if kind == "f32":
        check_f32(y, ref, oracle.abs_prefix(x))
    else:
        assert np.array_equal(y, ref)


@pytest.mark.parametrize("variant", [0, 1, 2, 3, 4, 5, 6, 7])
def test_compact_kernel_variants(variant):
    """Every compaction kernel (persistent with 8 or 16 compute warps, one tile
    per CTA, persistent with packed 16-byte stores, persistent with 4 + 2 or
    2 + 4 stages, persistent with a lag of 6 or 4 tiles) gives the oracle's result,
    for ragged sizes, all predicates and both count widths' paths."""
    import stream_compaction_gb300 as sc
    assert sc.sc_set_compact_variant(variant) == sc.SC_OK
    try:
        rng = np.random.default_rng(variant)
        for n in (8192, 8193, 16384 * 3 + 5, 1000003, (1 << 22) + 7):
            for dtype in ("i32", "u32", "f32"):
                if dtype == "i32":
                    x = rng.integers(-(1 << 20), 1 << 20, n).astype(np.int32)
                    thr = 0
                elif dtype == "u32":
                    x = rng.integers(0, 1 << 32, n, dtype=np.uint64).astype(np.uint32)
                    thr = float(1 << 31)
                else:
                    x = rng.uniform(-1, 1, n).astype(np.float32)
                    thr = 0.25
                for pred in ("gt", "le", "ne"):
                    out, c, full = gpu_compact(x, pred, thr)
                    ref, rc = oracle.compact(x, pred, thr)
                    assert c == rc and np.array_equal(out.view(np.int32), ref.view(np.int32)), (n, dtype, pred)
                    if c < n:
                        assert np.all(full[c:n].view(np.int32) == -7)
    finally:
        sc.sc_set_compact_variant(0)


def _kept_pattern(kind, n, rng):
    """int32 inputs whose x > 0 pattern stresses the packed stores: every
    element kept (a warp's run fills its whole slot ring), none, one in a
    hundred, all but one in a hundred, alternating, and runs of random length."""
    if kind == "all":
        return np.arange(1, n + 1, dtype=np.int32)
    if kind == "none":
        return -np.arange(1, n + 1, dtype=np.int32)
    if kind == "sparse":
        return np.where(rng.random(n) < 0.01, 1, -1).astype(np.int32) * np.arange(1, n + 1, dtype=np.int32)
    if kind == "dense":
        return np.where(rng.random(n) < 0.99, 1, -1).astype(np.int32) * np.arange(1, n + 1, dtype=np.int32)
    if kind == "alternate":
        return np.where(np.arange(n) % 2 == 0, 1, -1).astype(np.int32) * np.arange(1, n + 1, dtype=np.int32)
    runs = np.repeat(rng.integers(0, 2, n // 7 + 1) * 2 - 1, 7)[:n]   # runs of 7 kept / 7 dropped, at random
    return (runs * np.arange(1, n + 1)).astype(np.int32)


@pytest.mark.parametrize("variant", [0, 1, 3, 4, 5, 6, 7])
@pytest.mark.parametrize("out_offset", [0, 1, 2, 3])
@pytest.mark.parametrize("kind", ["all", "none", "sparse", "dense", "alternate", "runs"])
def test_compact_persistent_output_alignment(variant, out_offset, kind):
    """The persistent kernels on 16-byte aligned inputs, with the output 0-3
    elements past a 16-byte boundary: each warp's run of kept elements starts
    anywhere inside an aligned group, so the packed path's partial end groups
    and its full 16-byte groups both occur.  Every kept element against the
    oracle, and nothing written past the count."""
    import stream_compaction_gb300 as sc
    assert sc.sc_set_compact_variant(variant) == sc.SC_OK
    try:
        rng = np.random.default_rng(out_offset * 10 + len(kind))
        for n in (8192, 8192 * 5 + 1, 8192 * 40 + 4097):
            x = _kept_pattern(kind, n, rng)
            out, c, full = gpu_compact(x, "gt", 0, offset=0, out_offset=out_offset)
            assert sc.sc_debug_last_path() == sc.SC_PATH_COMPACT_PERSISTENT
            ref, rc = oracle.compact(x, "gt", 0)
            assert c == rc and np.array_equal(out, ref), (n, kind)
            if c < n:
                assert np.all(full[c:n].view(np.int32) == -7), (n, kind)
    finally:
        sc.sc_set_compact_variant(0)
