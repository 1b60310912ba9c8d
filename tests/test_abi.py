"""The C-ABI library builds, loads, and exports every symbol include/sc_scan.h declares.

No compute calls: only the host-side argument checks, which return before any
CUDA call, are exercised here.
"""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sc_scan.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sc_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from stream_compaction_gb300 import build
    import stream_compaction_gb300 as sc
    build.build()
    return sc.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("sc_scan_inclusive", "sc_scan_exclusive", "sc_scan_batched", "sc_compact_if",
                     "sc_get_device_error", "sc_workspace_bytes"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    import ctypes
    import subprocess
    import stream_compaction_gb300 as sc
    out = subprocess.run(["nm", "-D", "--defined-only", sc.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (sc_\w+)", out))
    for name in declared_functions():
        assert name in exported, name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)
        assert name in sc.SIGNATURES, "binding lacks " + name


def test_host_side_argument_checks(lib):
    import stream_compaction_gb300 as sc
    # invalid enums and negative sizes are rejected before any CUDA call
    assert sc.sc_scan_inclusive(9, sc.SC_SUM, 0, 0, 10, 0) == sc.SC_ERR_INVALID
    assert sc.sc_scan_exclusive(sc.SC_I32, 8, 0, 0, 10, 0) == sc.SC_ERR_INVALID
    assert sc.sc_scan_exclusive(8, sc.SC_SUM, 0, 0, 10, 0) == sc.SC_ERR_INVALID
    assert sc.sc_scan_exclusive(sc.SC_I32, sc.SC_SUM, 0, 0, -1, 0) == sc.SC_ERR_INVALID
    # unsupported operator/dtype pairs
    assert sc.sc_scan_inclusive(sc.SC_F32, sc.SC_PROD, 0, 0, 0, 0) == sc.SC_ERR_UNSUPPORTED
    assert sc.sc_scan_inclusive(sc.SC_F64, sc.SC_XOR, 0, 0, 0, 0) == sc.SC_ERR_UNSUPPORTED
    assert sc.sc_scan_inclusive(sc.SC_I32, sc.SC_COMPOSE, 0, 0, 0, 0) == sc.SC_ERR_UNSUPPORTED
    assert sc.sc_scan_inclusive(sc.SC_MAXCOUNT_I32, sc.SC_MIN, 0, 0, 0, 0) == sc.SC_ERR_UNSUPPORTED
    assert sc.sc_scan_batched(sc.SC_AFFINE_U32, sc.SC_AND, 1, 0, 0, 0, 0, 0) == sc.SC_ERR_UNSUPPORTED
    # every listed (dtype, op) pair passes the host checks (n == 0: no launch)
    for dt in (sc.SC_I32, sc.SC_U32, sc.SC_I64, sc.SC_U64):
        for op in (sc.SC_SUM, sc.SC_MAX, sc.SC_MIN, sc.SC_PROD, sc.SC_AND, sc.SC_OR, sc.SC_XOR):
            assert sc.sc_scan_inclusive(dt, op, 0, 0, 0, 0) == sc.SC_OK, (dt, op)
    for dt in (sc.SC_F32, sc.SC_F64):
        for op in (sc.SC_SUM, sc.SC_MAX, sc.SC_MIN):
            assert sc.sc_scan_exclusive(dt, op, 0, 0, 0, 0) == sc.SC_OK, (dt, op)
    assert sc.sc_scan_exclusive(sc.SC_MAXCOUNT_I32, sc.SC_MAX, 0, 0, 0, 0) == sc.SC_OK
    # 8-byte types need 8-byte alignment
    assert sc.sc_scan_inclusive(sc.SC_I64, sc.SC_SUM, 0x1004, 0x2000, 5, 0) == sc.SC_ERR_INVALID
    # empty input is a no-op; null pointers with n > 0 are errors
    assert sc.sc_scan_inclusive(sc.SC_U32, sc.SC_SUM, 0, 0, 0, 0) == sc.SC_OK
    assert sc.sc_scan_inclusive(sc.SC_U32, sc.SC_SUM, 0, 0, 5, 0) == sc.SC_ERR_INVALID
    # misaligned element pointers and partial overlap
    assert sc.sc_scan_inclusive(sc.SC_U32, sc.SC_SUM, 0x1001, 0x2000, 5, 0) == sc.SC_ERR_INVALID
    assert sc.sc_scan_inclusive(sc.SC_U32, sc.SC_SUM, 0x1000, 0x1004, 5, 0) == sc.SC_ERR_INVALID
    assert sc.sc_scan_batched(sc.SC_I32, sc.SC_SUM, 1, 0x1000, 0x2000, -1, 4, 0) == sc.SC_ERR_INVALID
    # compaction: overlapping in/out, bad predicate, unsupported dtype
    assert sc.sc_compact_if(sc.SC_I32, 0x1000, 0x1008, 0x8000, 16, sc.SC_GT, 0.0, 0) == sc.SC_ERR_INVALID
    assert sc.sc_compact_if(sc.SC_I32, 0x1000, 0x9000, 0x8000, 16, 11, 0.0, 0) == sc.SC_ERR_INVALID
    assert sc.sc_compact_if(sc.SC_AFFINE_U32, 0x1000, 0x9000, 0x8000, 16, sc.SC_GT, 0.0, 0) == sc.SC_ERR_UNSUPPORTED
    assert sc.sc_compact_if(sc.SC_I32, 0x1000, 0x9000, 0, 16, sc.SC_GT, 0.0, 0) == sc.SC_ERR_INVALID
    # segmented scan: flags are required and must not overlap the output
    assert sc.sc_scan_segmented(sc.SC_I32, sc.SC_SUM, 1, 0x1000, 0, 0x9000, 16, 0) == sc.SC_ERR_INVALID
    assert sc.sc_scan_segmented(sc.SC_I32, sc.SC_SUM, 1, 0x1000, 0x9004, 0x9000, 16, 0) == sc.SC_ERR_INVALID
    assert sc.sc_scan_segmented(sc.SC_I32, sc.SC_COMPOSE, 1, 0x1000, 0x20000, 0x9000, 16, 0) == sc.SC_ERR_UNSUPPORTED
    assert sc.sc_scan_segmented(sc.SC_I64, sc.SC_XOR, 0, 0, 0, 0, 0, 0) == sc.SC_OK
    # histogram / bin offsets
    assert sc.sc_histogram(0x1000, 10, 0, 0x8000, 0) == sc.SC_ERR_INVALID            # no bins
    assert sc.sc_histogram(0x1000, -1, 5, 0x8000, 0) == sc.SC_ERR_INVALID
    assert sc.sc_histogram(0x1000, 10, 5, 0x8004, 0) == sc.SC_ERR_INVALID            # misaligned counts
    assert sc.sc_bin_offsets(0x1000, 10, 5, 0x1008, 0) == sc.SC_ERR_INVALID          # overlaps the bins
    assert sc.sc_bin_offsets(0x1002, 10, 5, 0x8000, 0) == sc.SC_ERR_INVALID          # misaligned bins
    # tuning and test hooks
    assert sc.sc_set_scan_variant(99) == sc.SC_ERR_INVALID
    assert sc.sc_set_radix_variant(-1) == sc.SC_ERR_INVALID
    assert sc.sc_set_radix_variant(6) == sc.SC_ERR_INVALID
    st, t, i, l = sc.sc_scan_variant_info(0)
    assert st == sc.SC_OK and l == 2 and t * i * 4 >= 16384  # persistent TMA kernel, >= 16 KiB tiles
    assert sc.sc_debug_set_lookback(-5, -1, 0, 0) == sc.SC_ERR_INVALID
    assert sc.sc_debug_set_lookback(-1, -1, 0, 0) == sc.SC_OK
    assert sc.sc_workspace_bytes(1 << 30) >= 8 * ((1 << 30) // 4096)
    assert "sm_103a" in sc.sc_version()
    assert "INVALID" in sc.status_string(sc.SC_ERR_INVALID)
