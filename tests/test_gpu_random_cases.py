"""Seeded random cases across the entry points, against the oracle: sizes near
the boundaries between kernel paths (one-tile kernel up to 2^22 elements,
8192-element tiles and 2-tile chunks of the persistent kernels), element
offsets that break 16-byte alignment, in-place calls, exclusive and
inclusive forms, head densities and operators.  Each case is exact (integers,
float max/min) or within the documented float bounds."""
import numpy as np
import pytest

import oracle
from gpu_helpers import check_f32, check_f64, ensure_lib, gpu_compact, gpu_scan, same_float
from test_gpu_ops import make_input
from test_gpu_segmented import gpu_segmented

pytestmark = pytest.mark.gpu

OPS = [("u32", "sum"), ("i32", "max"), ("f32", "sum"), ("i32", "min"), ("u32", "xor"), ("u32", "prod"),
       ("f32", "max"), ("i64", "sum"), ("f64", "sum"), ("u64", "min"), ("maxcount", "maxcount")]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def _size(rng):
    base = int(rng.choice([8192, 16384, 1 << 21, 1 << 22, 3 * 16384, 4096, 64 * 16384]))
    return max(1, base * int(rng.integers(1, 3)) + int(rng.integers(-70, 70)))


def _check(kind, op, x, y, ref, scale):
    if kind == "f32" and op == "sum":
        check_f32(y, ref, scale)
    elif kind == "f64" and op == "sum":
        check_f64(y, ref, scale)
    elif kind in ("f32", "f64"):
        assert same_float(y, ref)
    else:
        assert np.array_equal(y, ref)


@pytest.mark.parametrize("case", range(24))
def test_random_scan(case):
    rng = np.random.default_rng(1000 + case)
    kind, op = OPS[case % len(OPS)]
    n = _size(rng)
    x = make_input(kind, op, n, seed=case)
    ex = bool(rng.integers(0, 2))
    off = int(rng.integers(0, 2)) * (2 if kind == "maxcount" else 1)
    inplace = bool(rng.integers(0, 2))
    y = gpu_scan(x, op, ex, offset=off, inplace=inplace)
    scale = oracle.abs_prefix(x) if op == "sum" and kind in ("f32", "f64") else None
    _check(kind, op, x, y, oracle.scan(x, op, ex), scale)


@pytest.mark.parametrize("case", range(24))
def test_random_segmented(case):
    rng = np.random.default_rng(2000 + case)
    kind, op = OPS[case % len(OPS)]
    n = _size(rng)
    x = make_input(kind, op, n, seed=case + 50)
    density = float(rng.choice([0.0, 1e-5, 1e-3, 0.05, 1.0]))
    h = (rng.random(n) < density).astype(np.uint8) * rng.integers(1, 256, n).astype(np.uint8)
    ex = bool(rng.integers(0, 2))
    off = int(rng.integers(0, 2)) * (2 if kind == "maxcount" else 1)
    hoff = int(rng.choice([0, 0, 1, 16]))
    y = gpu_segmented(x, h, op, ex, offset=off, hoff=hoff)
    scale = None
    if op == "sum" and kind in ("f32", "f64"):
        scale = oracle.scan_segmented(np.abs(x.astype(np.float64)), h, "sum", False)
    _check(kind, op, x, y, oracle.scan_segmented(x, h, op, ex), scale)


@pytest.mark.parametrize("case", range(12))
def test_random_compaction(case):
    rng = np.random.default_rng(3000 + case)
    kind = ["i32", "u32", "f32"][case % 3]
    n = _size(rng)
    if kind == "f32":
        x = rng.uniform(-1, 1, n).astype(np.float32)
    else:
        x = rng.integers(-1000, 1000, n).astype(np.int32 if kind == "i32" else np.uint32)
    pred = str(rng.choice(["gt", "ge", "lt", "le", "eq", "ne"]))
    t = float(rng.choice([0.0, 0.5, -3.0, 7.0]))
    off = int(rng.integers(0, 2))
    got, c, _ = gpu_compact(x, pred, t, offset=off)
    ref, rc = oracle.compact(x, pred, t)
    assert c == rc
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


ROW_OPS = [("i32", "sum"), ("u32", "sum"), ("i32", "max"), ("f32", "sum"), ("u32", "xor"), ("f32", "max"),
           ("i64", "sum"), ("affine", "affine")]


@pytest.mark.parametrize("case", range(24))
def test_random_batched_rows(case):
    """Batched rows with random row lengths (dividing 8192 or not, shorter and
    longer than a tile), row counts (one tile up to several tiles per CTA),
    element offsets and in-place calls: the rows kernel, its ragged form, the
    segmented kernels and the one-tile kernel, each against the oracle."""
    import stream_compaction_gb300 as sc
    from gpu_helpers import CODE, OPC, dev_buffer, stream, to_device, to_host
    rng = np.random.default_rng(4000 + case)
    kind, op = ROW_OPS[case % len(ROW_OPS)]
    cols = int(rng.choice([1, 3, 16, 31, 33, 64, 100, 1000, 2047, 2048, 4095, 8191, 8192, 12289]))
    n_target = int(rng.choice([8192, 65536, 1 << 20, 3 << 20]))
    rows = max(1, n_target // cols + int(rng.integers(0, 3)))
    if kind == "affine":
        x = np.random.default_rng(case + 90).integers(0, 1 << 32, (rows, cols, 2), dtype=np.uint64).astype(np.uint32)
    else:
        x = make_input(kind, op, rows * cols, seed=case + 90).reshape(rows, cols)
    ex = bool(rng.integers(0, 2))
    off = int(rng.integers(0, 2)) * (2 if kind == "affine" else 1)
    inplace = bool(rng.integers(0, 2))
    _, xin = to_device(x, off)
    xout = xin if inplace else dev_buffer(xin.numel(), xin.dtype, off)[1]
    st = sc.sc_scan_batched(CODE[kind], OPC[op], int(ex), xin.data_ptr(), xout.data_ptr(), rows, cols, stream())
    assert st == sc.SC_OK, sc.status_string(st)
    assert sc.sc_get_device_error(stream()) == sc.SC_OK
    y = to_host(xout, x)
    ref = oracle.scan_batched(x, op, ex)
    what = "%s %s rows=%d cols=%d excl=%d off=%d inplace=%d" % (kind, op, rows, cols, ex, off, inplace)
    if kind == "f32" and op == "sum":
        s_abs = np.stack([oracle.abs_prefix(r) for r in x])
        check_f32(y.reshape(-1), ref.reshape(-1), s_abs.reshape(-1), what)
    elif kind != "f32":
        assert np.array_equal(y, ref), what
    else:
        assert same_float(y, ref), what

