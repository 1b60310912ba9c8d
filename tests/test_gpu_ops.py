"""GPU parity for the operators beyond sum / max / compose: min, product, bitwise
and / or / xor on 32- and 64-bit integers, 64-bit sums, float max / min, float64
sums and (max, count) pairs, each against the CPU oracle.

Integer operators, float max / min and (max, count) must match bit for bit
(float NaN outputs: both NaN); float64 sums must lie within the bound
documented in include/sc_scan.h (gpu_helpers.check_f64).  Sizes cover one
element, ragged tiles of both element sizes, the short-scan path (n <= 2^22)
and the persistent kernel (larger n) with a ragged last chunk.
"""
import numpy as np
import pytest

import oracle
from gpu_helpers import check_f64, ensure_lib, gpu_batched, gpu_scan, same_float, stream, to_device

pytestmark = pytest.mark.gpu

M32, M64 = 1 << 32, 1 << 64

CASES = [("i32", "min"), ("u32", "max"), ("u32", "min"), ("i32", "prod"), ("u32", "prod"), ("i32", "and"),
         ("u32", "or"), ("i32", "xor"), ("u32", "xor"), ("i64", "sum"), ("u64", "sum"), ("i64", "prod"),
         ("u64", "prod"), ("u64", "and"), ("i64", "or"), ("u64", "xor"), ("i64", "max"), ("i64", "min"),
         ("u64", "max"), ("u64", "min"), ("f32", "max"), ("f32", "min"), ("f64", "sum"), ("f64", "max"),
         ("f64", "min"), ("maxcount", "maxcount")]
SIZES = [1, 2, 31, 33, 2047, 2049, 4097, 3 * 4096 + 5, 100003, (1 << 21) + 1, (1 << 22) + 1, 3 * (1 << 21) + 77]

_NP = {"i32": np.int32, "u32": np.uint32, "i64": np.int64, "u64": np.uint64, "f32": np.float32, "f64": np.float64}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def make_input(kind, op, n, seed):
    """Inputs that keep each operator's running value changing: odd factors for
    products (a zero only near the end), dense bits for and, sparse bits for or,
    a trend with rare extreme spikes for integer max / min, and NaNs, signed
    zeros and infinities for float max and min."""
    rng = np.random.default_rng(seed)
    if kind == "maxcount":
        return np.stack([rng.integers(-40, 40, n), rng.integers(0, 4, n)], axis=1).astype(np.int32)
    dt = np.dtype(_NP[kind])
    if dt.kind == "f":
        if op == "sum":
            return (rng.uniform(-1, 1, n) * 10.0 ** rng.integers(-6, 6, n)).astype(dt)
        trend = np.cumsum(rng.uniform(-1, 1.5, n))   # rising on average: new records often
        x = (trend if op == "max" else -trend).astype(dt)
        special = np.array([-0.0, 0.0, np.inf, -np.inf, 1e30, -1e30], dtype=dt)
        k = max(1, n // 5000)
        x[rng.integers(n - n // 10 - 1, n, k)] = special[rng.integers(0, special.size, k)]  # in the last tenth
        if n > 10:
            x[n // 2] = -0.0
            x[n // 2 + 1] = 0.0
            x[n - n // 5] = np.nan                  # NaN from here on
        return x
    bits = 8 * dt.itemsize
    u = np.dtype("u%d" % dt.itemsize)
    r = rng.integers(0, 1 << 62, n, dtype=np.int64).astype(np.uint64)
    r = (r << np.uint64(2)) | rng.integers(0, 4, n, dtype=np.uint64)  # full 64 random bits
    if op == "prod":
        r = r | np.uint64(1)                       # odd factors: the product never sticks at 0
        if n > 100:
            r[n - 1 - n // 100] = 0
    elif op == "and":
        clear = rng.random(n) < 2.0 / max(n, 1) * bits
        r = np.where(clear, ~(np.uint64(1) << (r % np.uint64(bits))), ~np.uint64(0))
    elif op == "or":
        r = np.where(rng.random(n) < 2.0 / max(n, 1) * bits, np.uint64(1) << (r % np.uint64(bits)), np.uint64(0))
    elif op in ("max", "min"):
        # a trend away from the type's far end (new records all the time), and in
        # the last tenth rare full-range values
        info = np.iinfo(dt)
        walk = np.abs(np.cumsum(rng.integers(-3, 6, n))).astype(dt)
        base = (np.array(info.min, dt) + walk) if op == "max" else (np.array(info.max, dt) - walk)
        spike = (np.arange(n) > 0.9 * n) & (rng.random(n) > 0.995)
        return np.where(spike, r.astype(u).view(dt), base)
    return r.astype(u).view(dt)


def check(kind, op, x, y, ref):
    if kind == "f64" and op == "sum":
        check_f64(y, ref, oracle.abs_prefix(x))
    elif kind in ("f32", "f64"):
        assert same_float(y, ref)
    else:
        assert np.array_equal(y, ref)


@pytest.mark.parametrize("kind,op", CASES)
@pytest.mark.parametrize("exclusive", [False, True])
@pytest.mark.parametrize("n", SIZES)
def test_scan_more_ops(kind, op, exclusive, n):
    x = make_input(kind, op, n, seed=n * 13 + len(op))
    y = gpu_scan(x, op, exclusive)
    check(kind, op, x, y, oracle.scan(x, op, exclusive))


@pytest.mark.parametrize("kind,op", CASES)
def test_more_ops_unaligned_and_inplace(kind, op):
    n = 5 * 4096 + 7
    x = make_input(kind, op, n, seed=77)
    off = 2 if kind == "maxcount" else 1      # element-aligned, not 16-byte aligned
    for ex in (False, True):
        ref = oracle.scan(x, op, ex)
        for y in (gpu_scan(x, op, ex, offset=off), gpu_scan(x, op, ex, inplace=True),
                  gpu_scan(x, op, ex, offset=off, inplace=True)):
            check(kind, op, x, y, ref)


@pytest.mark.parametrize("kind,op", [("u32", "xor"), ("i64", "sum"), ("i64", "min"), ("f32", "max"),
                                     ("f64", "sum"), ("maxcount", "maxcount"), ("u64", "prod")])
@pytest.mark.parametrize("shape", [(1, 5000), (7, 3), (100, 17), (5, 4096), (3, 4097), (64, 8195)])
def test_batched_more_ops(kind, op, shape):
    rows, cols = shape
    x = make_input(kind, op, rows * cols, seed=rows * 31 + cols)
    x = x.reshape((rows, cols) + x.shape[1:])
    for ex in (False, True):
        y = gpu_batched(x, op, ex)
        ref = oracle.scan_batched(x, op, ex)
        if kind == "f64" and op == "sum":
            for r in range(rows):
                check_f64(y[r], ref[r], oracle.abs_prefix(x[r]))
        else:
            check(kind, op, x, y, ref)


def test_float_max_min_special_values():
    """NaN propagates from its position on; of equal values (-0.0, +0.0) the earlier wins."""
    for dt in (np.float32, np.float64):
        x = np.array([-0.0, 0.0, 1.0, -np.inf, np.inf, 2.0, np.nan, 5.0], dtype=dt)
        for op in ("max", "min"):
            for ex in (False, True):
                assert same_float(gpu_scan(x, op, ex), oracle.scan(x, op, ex)), (dt, op, ex)
        y = gpu_scan(x, "max", False)
        assert np.signbit(y[0]) and np.signbit(y[1])      # -0.0 first, then +0.0 does not replace it
        assert np.isnan(y[6:]).all()


def test_scan_host_more_ops():
    import torch
    import stream_compaction_gb300 as sc
    n = (1 << 23) + 4099                    # two chunks of the host pipeline (64 MiB of float64 each)
    for kind, op in (("f64", "sum"), ("u64", "xor"), ("i32", "min")):
        x = make_input(kind, op, n, seed=5)
        xt = torch.from_numpy(x.view(np.int64) if x.dtype.itemsize == 8 else x.view(np.int32)).pin_memory()
        yt = torch.empty_like(xt).pin_memory()
        from gpu_helpers import CODE, OPC
        st = sc.sc_scan_host(CODE[kind], OPC[op], 1, xt.data_ptr(), yt.data_ptr(), n, stream())
        assert st == sc.SC_OK
        check(kind, op, x, yt.numpy().view(x.dtype), oracle.scan(x, op, True))


def test_unsupported_pairs_and_entry_points():
    import stream_compaction_gb300 as sc
    _, xin = to_device(np.arange(10, dtype=np.int64))
    _, xout = to_device(np.zeros(10, dtype=np.int64))
    p, q, s = xin.data_ptr(), xout.data_ptr(), stream()
    for dt, op in ((sc.SC_F32, sc.SC_PROD), (sc.SC_F64, sc.SC_XOR), (sc.SC_AFFINE_U32, sc.SC_MIN),
                   (sc.SC_MAXCOUNT_I32, sc.SC_SUM), (sc.SC_I64, sc.SC_COMPOSE)):
        assert sc.sc_scan_inclusive(dt, op, p, q, 10, s) == sc.SC_ERR_UNSUPPORTED
    # the comparison variant and the no-allocation entry point keep the first four operators
    assert sc.sc_scan_hierarchical(sc.SC_I64, sc.SC_SUM, 1, p, q, 10, s) == sc.SC_ERR_UNSUPPORTED
    assert sc.sc_hier_workspace_bytes(sc.SC_I64, 1000) == 0
    assert sc.sc_scan_noalloc(sc.SC_I64, sc.SC_SUM, 1, p, q, 10, s) == sc.SC_ERR_UNSUPPORTED
    # the compaction keeps its three dtypes
    cnt = to_device(np.zeros(1, dtype=np.int64))[1]
    assert sc.sc_compact_if(sc.SC_I64, p, q, cnt.data_ptr(), 10, sc.SC_GT, 0.0, s) == sc.SC_ERR_UNSUPPORTED


@pytest.mark.parametrize("name", ["int64_exsum_n2^27", "float64_exsum_n2^26", "int32_min_n2^27", "uint32_xor_n2^27",
                                  "float32_max_n2^26", "maxcount_i32_n2^26"])
def test_added_operator_workloads(name):
    """The benchmark workloads of the added operators, at full size, against the oracle."""
    import torch
    from stream_compaction_gb300 import synth
    spec = synth.WORKLOADS[name]
    xt = synth.make_torch(spec, device="cuda")
    torch.cuda.synchronize()
    x = xt.cpu().numpy()
    kind = {"u64": "i64", "pm1_f64": "f64", "u32": "u32", "pm1": "f32", "maxcount": "maxcount"}[spec["kind"]]
    if kind == "u32" and spec["op"] == "min":
        x = x.view(np.int32)
    elif kind == "u32":
        x = x.view(np.uint32)
    ex = spec["op"] == "sum"
    y = gpu_scan(x, spec["op"], ex)
    check("f64" if kind == "f64" else kind, spec["op"], x, y, oracle.scan(x, spec["op"], ex))
