"""Helpers for the GPU parity tests: move numpy inputs to the device, call the
library through its C-named binding, bring results back."""
from __future__ import annotations

import numpy as np

import stream_compaction_gb300 as sc

CODE = {"i32": sc.SC_I32, "u32": sc.SC_U32, "f32": sc.SC_F32, "affine": sc.SC_AFFINE_U32, "i64": sc.SC_I64,
        "u64": sc.SC_U64, "f64": sc.SC_F64, "maxcount": sc.SC_MAXCOUNT_I32}
OPC = {"sum": sc.SC_SUM, "max": sc.SC_MAX, "affine": sc.SC_COMPOSE, "min": sc.SC_MIN, "prod": sc.SC_PROD,
       "and": sc.SC_AND, "or": sc.SC_OR, "xor": sc.SC_XOR, "maxcount": sc.SC_MAX}


def ensure_lib():
    import torch
    from stream_compaction_gb300 import build
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build.build()
    return sc.load()


def stream():
    import torch
    return int(torch.cuda.current_stream().cuda_stream)


def dev_buffer(words: int, torch_dtype, offset: int = 0):
    """A device buffer with room for `words` elements starting `offset` elements in."""
    import torch
    base = torch.empty(words + offset + 8, dtype=torch_dtype, device="cuda")
    return base, base[offset:offset + words]


def to_device(x: np.ndarray, offset: int = 0):
    """Copy a numpy array (4- or 8-byte elements, any shape) into a flat device view;
    offset counts elements of that size."""
    import torch
    flat = np.ascontiguousarray(x).reshape(-1)
    if flat.dtype in (np.float32, np.float64):
        tdt = torch.float32 if flat.dtype == np.float32 else torch.float64
        src = torch.from_numpy(flat)
    elif flat.dtype.itemsize == 8:
        tdt = torch.int64
        src = torch.from_numpy(flat.view(np.int64))
    else:
        tdt = torch.int32
        src = torch.from_numpy(flat.view(np.int32))
    base, view = dev_buffer(flat.size, tdt, offset)
    view.copy_(src)
    return base, view


def to_host(view, like: np.ndarray) -> np.ndarray:
    import torch
    torch.cuda.synchronize()
    a = view.cpu().numpy()
    return a.view(like.dtype).reshape(like.shape) if a.dtype != like.dtype or a.shape != like.shape else a


def kind_of(x: np.ndarray, op: str) -> str:
    if op in ("affine", "maxcount"):
        return op
    return {np.dtype(np.int32): "i32", np.dtype(np.uint32): "u32", np.dtype(np.float32): "f32",
            np.dtype(np.int64): "i64", np.dtype(np.uint64): "u64", np.dtype(np.float64): "f64"}[x.dtype]


def gpu_scan(x: np.ndarray, op: str, exclusive: bool, offset: int = 0, inplace: bool = False,
             hierarchical: bool = False) -> np.ndarray:
    n = x.shape[0]
    _, xin = to_device(x, offset)
    if inplace:
        xout = xin
    else:
        _, xout = dev_buffer(xin.numel(), xin.dtype, (offset + 3) % 5 if offset else 0)
    k = kind_of(x, op)
    if hierarchical:
        st = sc.sc_scan_hierarchical(CODE[k], OPC[op], int(exclusive), xin.data_ptr(), xout.data_ptr(), n, stream())
    elif exclusive:
        st = sc.sc_scan_exclusive(CODE[k], OPC[op], xin.data_ptr(), xout.data_ptr(), n, stream())
    else:
        st = sc.sc_scan_inclusive(CODE[k], OPC[op], xin.data_ptr(), xout.data_ptr(), n, stream())
    assert st == sc.SC_OK, sc.status_string(st)
    assert sc.sc_get_device_error(stream()) == sc.SC_OK
    return to_host(xout, x)


def gpu_batched(x: np.ndarray, op: str, exclusive: bool) -> np.ndarray:
    rows, cols = x.shape[0], x.shape[1]
    _, xin = to_device(x)
    _, xout = dev_buffer(xin.numel(), xin.dtype)
    k = kind_of(x, op)
    st = sc.sc_scan_batched(CODE[k], OPC[op], int(exclusive), xin.data_ptr(), xout.data_ptr(), rows, cols, stream())
    assert st == sc.SC_OK, sc.status_string(st)
    assert sc.sc_get_device_error(stream()) == sc.SC_OK
    return to_host(xout, x)


def gpu_compact(x: np.ndarray, pred: str, threshold: float, offset: int = 0, out_offset: int | None = None):
    """Compaction through the C ABI; offset / out_offset: element offsets of the
    input and output buffers (16-byte aligned at 0)."""
    import torch
    n = x.shape[0]
    _, xin = to_device(x, offset)
    _, xout = dev_buffer(max(n, 1), xin.dtype, (1 if offset else 0) if out_offset is None else out_offset)
    (xout.view(torch.int32) if xout.dtype == torch.float32 else xout).fill_(-7)
    cnt = torch.full((1,), -1, dtype=torch.int64, device="cuda")
    st = sc.sc_compact_if(CODE[kind_of(x, "sum")], xin.data_ptr(), xout.data_ptr(), cnt.data_ptr(), n,
                          sc.PRED[pred], float(threshold), stream())
    assert st == sc.SC_OK, sc.status_string(st)
    assert sc.sc_get_device_error(stream()) == sc.SC_OK
    c = int(cnt.item())
    out = to_host(xout, np.zeros(max(n, 1), dtype=x.dtype))
    return out[:c].copy(), c, out


def check_f32(y_gpu: np.ndarray, y_ref: np.ndarray, abs_prefix: np.ndarray, what: str = ""):
    """Float32 sums: |y_gpu[i] - y_ref[i]| <= 1e-5 * sum_{k<=i} |x[k]| for every i."""
    err = np.abs(y_gpu.astype(np.float64) - y_ref)
    bound = 1e-5 * abs_prefix
    bad = np.nonzero(err > bound)[0]
    assert bad.size == 0, "%s: %d elements outside the bound, first at %d (err %g, bound %g)" % (
        what, bad.size, bad[0], err[bad[0]], bound[bad[0]])
    return float(np.max(err / np.maximum(abs_prefix, 1e-300))) if err.size else 0.0


def check_f64(y_gpu: np.ndarray, y_ref: np.ndarray, abs_prefix: np.ndarray, what: str = ""):
    """Float64 sums: |y_gpu[i] - y_ref[i]| <= (16 * ceil(n/2048) + 64) * 2^-53 * sum_{k<=i} |x[k]|.

    Each output is a sum of partial sums rounded along its dependency chain:
    a tile's prefix comes from an earlier tile's prefix plus a fold of the
    aggregates in between (at most 16 roundings deep: a 5-level warp tree, up to
    8 serial folds per lane, 3 combines), and a chain has at most one such hop
    per tile (tiles hold at least 2048 float64 elements); inside a tile there
    are fewer than 64 more roundings.  Each rounding is a relative error of at
    most 2^-53 of a partial sum no larger than sum |x|.  The oracle itself is
    within 4 * 2^-53 of the exact prefix."""
    n = y_ref.size
    bound = (16 * -(-n // 2048) + 64) * 2.0 ** -53 * abs_prefix
    err = np.abs(y_gpu - y_ref)
    bad = np.nonzero(err > bound)[0]
    assert bad.size == 0, "%s: %d elements outside the bound, first at %d (err %g, bound %g)" % (
        what, bad.size, bad[0], err[bad[0]], bound[bad[0]])


def same_float(a: np.ndarray, b: np.ndarray) -> bool:
    """Equal bit for bit, or both NaN (the exact float max/min scans)."""
    bits = np.uint32 if a.dtype == np.float32 else np.uint64
    return bool(np.all((a.view(bits) == b.view(bits)) | (np.isnan(a) & np.isnan(b))))
