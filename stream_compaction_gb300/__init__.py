"""GB300-native (sm_103a) device-wide scan and stream compaction.

Thin Python binding over the C ABI of ``libsc_gb300.so`` (declared in
``include/sc_scan.h``).  Two layers, both argument marshalling only:

* ``sc_*`` functions with the C names and the C argument order (integer
  device pointers, element counts, a raw ``cudaStream_t``);
* tensor helpers (``scan_inclusive``, ``scan_exclusive``, ``scan_batched``,
  ``compact_if``, ``scan_hierarchical``, ``scan_host``) that take torch CUDA
  tensors and the current torch stream.

Every step of the computation runs in the library's CUDA kernels.  There is no
CPU fallback: if the library has not been built (``python -m
stream_compaction_gb300.build``) the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsc_gb300.so")

# enums of include/sc_scan.h
SC_I32, SC_U32, SC_F32, SC_AFFINE_U32, SC_I64, SC_U64, SC_F64, SC_MAXCOUNT_I32 = 0, 1, 2, 3, 4, 5, 6, 7
SC_SUM, SC_MAX, SC_COMPOSE, SC_MIN, SC_PROD, SC_AND, SC_OR, SC_XOR = 0, 1, 2, 3, 4, 5, 6, 7
SC_GT, SC_GE, SC_LT, SC_LE, SC_EQ, SC_NE = 0, 1, 2, 3, 4, 5
SC_OK, SC_ERR_INVALID, SC_ERR_UNSUPPORTED, SC_ERR_WORKSPACE, SC_ERR_CUDA, SC_ERR_LOOKBACK_TIMEOUT, SC_ERR_INTERNAL = \
    range(7)

PRED = {"gt": SC_GT, "ge": SC_GE, "lt": SC_LT, "le": SC_LE, "eq": SC_EQ, "ne": SC_NE}

# every exported entry point and its ctypes signature
_P, _I64, _INT, _SZ, _D, _U32, _U64 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t,
                                      ctypes.c_double, ctypes.c_uint32, ctypes.c_uint64)
SIGNATURES = {
    "sc_version": ([], ctypes.c_char_p),
    "sc_status_string": ([_INT], ctypes.c_char_p),
    "sc_workspace_bytes": ([_I64], _SZ),
    "sc_set_workspace": ([_P, _SZ, _P], _INT),
    "sc_scan_inclusive": ([_INT, _INT, _P, _P, _I64, _P], _INT),
    "sc_scan_exclusive": ([_INT, _INT, _P, _P, _I64, _P], _INT),
    "sc_scan_batched": ([_INT, _INT, _INT, _P, _P, _I64, _I64, _P], _INT),
    "sc_compact_if": ([_INT, _P, _P, _P, _I64, _INT, _D, _P], _INT),
    "sc_scan_hierarchical": ([_INT, _INT, _INT, _P, _P, _I64, _P], _INT),
    "sc_hier_workspace_bytes": ([_INT, _I64], _SZ),
    "sc_scan_host": ([_INT, _INT, _INT, _P, _P, _I64, _P], _INT),
    "sc_scan_noalloc": ([_INT, _INT, _INT, _P, _P, _I64, _P], _INT),
    "sc_scan_segmented": ([_INT, _INT, _INT, _P, _P, _P, _I64, _P], _INT),
    "sc_histogram": ([_P, _I64, _I64, _P, _P], _INT),
    "sc_radix_pass_u32": ([_P, _P, _I64, _INT, _INT, _P], _INT),
    "sc_radix_sort_u32": ([_P, _P, _P, _I64, _P], _INT),
    "sc_bin_offsets": ([_P, _I64, _I64, _P, _P], _INT),
    "sc_get_device_error": ([_P], _INT),
    "sc_release_stream": ([_P], _INT),
    "sc_scan_noalloc_error": ([_P], _INT),
    "sc_debug_last_path": ([], _INT),
    "sc_launch_count": ([], _U64),
    "sc_set_scan_variant": ([_INT], _INT),
    "sc_set_compact_variant": ([_INT], _INT),
    "sc_set_status_stride": ([_INT], _INT),
    "sc_set_radix_variant": ([_INT], _INT),
    "sc_scan_variant_info": ([_INT, ctypes.POINTER(_INT), ctypes.POINTER(_INT), ctypes.POINTER(_INT)], _INT),
    "sc_debug_set_lookback": ([_I64, _I64, _U32, _U64], _INT),
    "sc_debug_lookback_stats": ([_P, ctypes.POINTER(_U64)], _INT),
}

_lock = threading.Lock()
_cdll = None


class ScanError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s" % (where, status_string(status)))


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libsc_gb300.so (raises if it has not been built)."""
    global _cdll
    with _lock:
        if _cdll is None:
            if not os.path.exists(path):
                raise RuntimeError("libsc_gb300.so is not built (%s); run "
                                   "`python -m stream_compaction_gb300.build` on a machine with nvcc" % path)
            lib = ctypes.CDLL(path)
            for name, (args, res) in SIGNATURES.items():
                f = getattr(lib, name)
                f.argtypes = args
                f.restype = res
            _cdll = lib
        return _cdll


def _check(status: int, where: str) -> None:
    if status != SC_OK:
        raise ScanError(status, where)


# ------------------------------------------------------------ C-named layer
def sc_version() -> str:
    return load().sc_version().decode()


def status_string(status: int) -> str:
    try:
        return load().sc_status_string(status).decode()
    except RuntimeError:
        return "status %d" % status


def sc_workspace_bytes(n: int) -> int:
    return load().sc_workspace_bytes(n)


def sc_set_workspace(d_ws: int, nbytes: int, stream: int) -> int:
    return load().sc_set_workspace(d_ws, nbytes, stream)


def sc_scan_inclusive(dtype: int, op: int, d_in: int, d_out: int, n: int, stream: int) -> int:
    return load().sc_scan_inclusive(dtype, op, d_in, d_out, n, stream)


def sc_scan_exclusive(dtype: int, op: int, d_in: int, d_out: int, n: int, stream: int) -> int:
    return load().sc_scan_exclusive(dtype, op, d_in, d_out, n, stream)


def sc_scan_batched(dtype: int, op: int, exclusive: int, d_in: int, d_out: int, rows: int, cols: int,
                    stream: int) -> int:
    return load().sc_scan_batched(dtype, op, exclusive, d_in, d_out, rows, cols, stream)


def sc_compact_if(dtype: int, d_in: int, d_out: int, d_count: int, n: int, pred: int, threshold: float,
                  stream: int) -> int:
    return load().sc_compact_if(dtype, d_in, d_out, d_count, n, pred, threshold, stream)


def sc_scan_hierarchical(dtype: int, op: int, exclusive: int, d_in: int, d_out: int, n: int, stream: int) -> int:
    return load().sc_scan_hierarchical(dtype, op, exclusive, d_in, d_out, n, stream)


def sc_hier_workspace_bytes(dtype: int, n: int) -> int:
    return load().sc_hier_workspace_bytes(dtype, n)


def sc_scan_host(dtype: int, op: int, exclusive: int, h_in: int, h_out: int, n: int, stream: int) -> int:
    return load().sc_scan_host(dtype, op, exclusive, h_in, h_out, n, stream)


def sc_scan_noalloc(dtype: int, op: int, exclusive: int, d_in: int, d_out: int, n: int, stream: int) -> int:
    return load().sc_scan_noalloc(dtype, op, exclusive, d_in, d_out, n, stream)


def sc_scan_segmented(dtype: int, op: int, exclusive: int, d_in: int, d_heads: int, d_out: int, n: int,
                      stream: int) -> int:
    return load().sc_scan_segmented(dtype, op, exclusive, d_in, d_heads, d_out, n, stream)


SC_NOALLOC_MAX_N = 1 << 27


def sc_get_device_error(stream: int) -> int:
    return load().sc_get_device_error(stream)


def sc_launch_count() -> int:
    return load().sc_launch_count()


def sc_release_stream(stream: int) -> int:
    return load().sc_release_stream(stream)


def sc_scan_noalloc_error(stream: int) -> int:
    return load().sc_scan_noalloc_error(stream)


# kernel families reported by sc_debug_last_path
(SC_PATH_NONE, SC_PATH_SCAN_ONE_TILE, SC_PATH_SCAN_PERSISTENT, SC_PATH_SEGSCAN_PERSISTENT,
 SC_PATH_COMPACT_PERSISTENT, SC_PATH_COMPACT_ONE_TILE, SC_PATH_ROWS_PERSISTENT) = range(7)


def sc_debug_last_path() -> int:
    return load().sc_debug_last_path()


def sc_set_scan_variant(variant: int) -> int:
    return load().sc_set_scan_variant(variant)


def sc_set_compact_variant(variant: int) -> int:
    return load().sc_set_compact_variant(variant)


def sc_set_status_stride(nbytes: int) -> int:
    return load().sc_set_status_stride(nbytes)


def sc_set_radix_variant(variant: int) -> int:
    return load().sc_set_radix_variant(variant)


def sc_scan_variant_info(variant: int):
    t, i, l = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    st = load().sc_scan_variant_info(variant, ctypes.byref(t), ctypes.byref(i), ctypes.byref(l))
    return st, t.value, i.value, l.value


def sc_debug_set_lookback(stall_tile: int, delay_tile: int, delay_ns: int, timeout_ns: int) -> int:
    return load().sc_debug_set_lookback(stall_tile, delay_tile, delay_ns, timeout_ns)


def sc_debug_lookback_stats(stream: int):
    buf = (_U64 * 8)()
    st = load().sc_debug_lookback_stats(stream, buf)
    return st, list(buf)


# ------------------------------------------------------------ tensor layer
def _stream(stream=None) -> int:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


_PAIR_OPS = {"affine": SC_AFFINE_U32, "maxcount": SC_MAXCOUNT_I32}


def _dtype_code(x, op: str) -> int:
    import torch
    if op in _PAIR_OPS:
        if x.dtype not in (torch.int32, torch.uint32) or x.dim() < 1 or x.shape[-1] != 2:
            raise ValueError("%s scan expects an int32/uint32 tensor of shape (..., 2)" % op)
        return _PAIR_OPS[op]
    m = {torch.int32: SC_I32, torch.float32: SC_F32, torch.int64: SC_I64, torch.float64: SC_F64}
    for name, code in (("uint32", SC_U32), ("uint64", SC_U64)):
        if hasattr(torch, name):
            m[getattr(torch, name)] = code
    if x.dtype not in m:
        raise ValueError("unsupported dtype %s" % x.dtype)
    return m[x.dtype]


# affine: (a, b) pairs composed; maxcount: (value, count) pairs (SC_MAXCOUNT_I32 with SC_MAX)
_OPS = {"sum": SC_SUM, "max": SC_MAX, "min": SC_MIN, "prod": SC_PROD, "and": SC_AND, "or": SC_OR, "xor": SC_XOR,
        "affine": SC_COMPOSE, "maxcount": SC_MAX}


def _prep(x, out, op):
    import torch
    if not x.is_cuda:
        raise ValueError("expected a CUDA tensor (use scan_host for host memory)")
    if not x.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    if out is None:
        out = torch.empty_like(x)
    if out.shape != x.shape or out.dtype != x.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor like x")
    n = x.numel() // 2 if op in _PAIR_OPS else x.numel()
    return out, n


def scan_inclusive(x, op: str = "sum", out=None, stream=None):
    """Inclusive scan of a 1-D CUDA tensor (affine, maxcount: shape (n, 2)).

    op: sum, max, min, prod, and, or, xor, affine, maxcount (see include/sc_scan.h
    for the dtypes each takes)."""
    out, n = _prep(x, out, op)
    _check(sc_scan_inclusive(_dtype_code(x, op), _OPS[op], x.data_ptr(), out.data_ptr(), n, _stream(stream)),
           "sc_scan_inclusive")
    return out


def scan_exclusive(x, op: str = "sum", out=None, stream=None):
    """Exclusive scan of a 1-D CUDA tensor (affine, maxcount: shape (n, 2))."""
    out, n = _prep(x, out, op)
    _check(sc_scan_exclusive(_dtype_code(x, op), _OPS[op], x.data_ptr(), out.data_ptr(), n, _stream(stream)),
           "sc_scan_exclusive")
    return out


def scan_batched(x, op: str = "sum", exclusive: bool = True, out=None, stream=None):
    """Row-wise scans of a row-major (rows, cols) CUDA tensor ((rows, cols, 2) for the pair ops)."""
    out, _ = _prep(x, out, op)
    rows, cols = x.shape[0], x.shape[1]
    _check(sc_scan_batched(_dtype_code(x, op), _OPS[op], int(exclusive), x.data_ptr(), out.data_ptr(), rows, cols,
                           _stream(stream)), "sc_scan_batched")
    return out


def scan_segmented(x, heads, op: str = "sum", exclusive: bool = True, out=None, stream=None):
    """Segmented scan of a 1-D CUDA tensor (pair ops: shape (n, 2)); heads is a
    CUDA uint8/bool tensor of n flags, nonzero where a segment starts."""
    import torch
    out, n = _prep(x, out, op)
    if not heads.is_cuda or heads.numel() != n or heads.dtype not in (torch.uint8, torch.bool, torch.int8):
        raise ValueError("heads must be a CUDA uint8/bool tensor with one flag per element")
    if not heads.is_contiguous():
        raise ValueError("heads must be contiguous")
    _check(sc_scan_segmented(_dtype_code(x, op), _OPS[op], int(exclusive), x.data_ptr(), heads.data_ptr(),
                             out.data_ptr(), n, _stream(stream)), "sc_scan_segmented")
    return out


def sc_histogram(d_bins: int, n: int, nbins: int, d_counts: int, stream: int) -> int:
    return load().sc_histogram(d_bins, n, nbins, d_counts, stream)


def sc_bin_offsets(d_bins: int, n: int, nbins: int, d_offsets: int, stream: int) -> int:
    return load().sc_bin_offsets(d_bins, n, nbins, d_offsets, stream)


def sc_radix_pass_u32(d_in: int, d_out: int, n: int, shift: int, bits: int, stream: int) -> int:
    return load().sc_radix_pass_u32(d_in, d_out, n, shift, bits, stream)


def sc_radix_sort_u32(d_in: int, d_out: int, d_tmp: int, n: int, stream: int) -> int:
    return load().sc_radix_sort_u32(d_in, d_out, d_tmp, n, stream)


def radix_sort(keys, out=None, tmp=None, stream=None):
    """Ascending sort of a CUDA uint32 (or int32 holding uint32 bits) tensor."""
    import torch
    if not keys.is_cuda or keys.element_size() != 4 or not keys.is_contiguous():
        raise ValueError("keys must be a contiguous CUDA tensor of 4-byte unsigned keys")
    out = torch.empty_like(keys) if out is None else out
    tmp = torch.empty_like(keys) if tmp is None else tmp
    _check(sc_radix_sort_u32(keys.data_ptr(), out.data_ptr(), tmp.data_ptr(), keys.numel(), _stream(stream)),
           "sc_radix_sort_u32")
    return out


def _bins_tensor(bins):
    import torch
    if not bins.is_cuda or bins.dtype != torch.int32 or not bins.is_contiguous():
        raise ValueError("bins must be a contiguous CUDA int32 tensor")
    return bins


def histogram(bins, nbins: int, out=None, stream=None):
    """int64 counts of each bin 0 .. nbins-1 in a CUDA int32 tensor (others skipped)."""
    import torch
    _bins_tensor(bins)
    if out is None:
        out = torch.empty(nbins, dtype=torch.int64, device=bins.device)
    _check(sc_histogram(bins.data_ptr(), bins.numel(), nbins, out.data_ptr(), _stream(stream)), "sc_histogram")
    return out


def bin_offsets(bins, nbins: int, out=None, stream=None):
    """int64 offsets (nbins + 1): exclusive scan of the histogram, total last
    (COO row indices -> CSR row pointers)."""
    import torch
    _bins_tensor(bins)
    if out is None:
        out = torch.empty(nbins + 1, dtype=torch.int64, device=bins.device)
    _check(sc_bin_offsets(bins.data_ptr(), bins.numel(), nbins, out.data_ptr(), _stream(stream)), "sc_bin_offsets")
    return out


def compact_if(x, pred: str = "gt", threshold: float = 0.0, out=None, count=None, stream=None):
    """Order-preserving compaction; returns (out, count) with count a 1-element int64 CUDA tensor.

    Only out[:count] is defined.  The count stays on the device (no host sync).
    """
    import torch
    out, n = _prep(x, out, "sum")
    if count is None:
        count = torch.empty(1, dtype=torch.int64, device=x.device)
    _check(sc_compact_if(_dtype_code(x, "sum"), x.data_ptr(), out.data_ptr(), count.data_ptr(), n, PRED[pred],
                         float(threshold), _stream(stream)), "sc_compact_if")
    return out, count


def scan_hierarchical(x, op: str = "sum", exclusive: bool = True, out=None, stream=None):
    """The multi-kernel hierarchical comparison variant (same results as scan_*)."""
    out, n = _prep(x, out, op)
    _check(sc_scan_hierarchical(_dtype_code(x, op), _OPS[op], int(exclusive), x.data_ptr(), out.data_ptr(), n,
                                _stream(stream)), "sc_scan_hierarchical")
    return out


def scan_host(x, op: str = "sum", exclusive: bool = True, out=None, stream=None):
    """Scan of a CPU tensor (pinned for overlap) through the library's host pipeline."""
    import torch
    if x.is_cuda or not x.is_contiguous():
        raise ValueError("scan_host expects a contiguous CPU tensor")
    if out is None:
        out = torch.empty_like(x, pin_memory=x.is_pinned())
    n = x.numel() // 2 if op in _PAIR_OPS else x.numel()
    _check(sc_scan_host(_dtype_code(x, op), _OPS[op], int(exclusive), x.data_ptr(), out.data_ptr(), n,
                        _stream(stream)), "sc_scan_host")
    return out


def get_device_error(stream=None) -> int:
    """Wait for the stream and return (and clear) its device error status."""
    return sc_get_device_error(_stream(stream))
