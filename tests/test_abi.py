"""C-ABI checks that need no GPU: the library builds for sm_103a, loads, and
exports every entry point that ``include/tb.h`` declares; host-side argument
checks answer before any device work."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tb.h")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"TB_API\s+[\w\s\*]+?\b(tb_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from sparse_voxel_grid_leaf_gb300 import _build
    path = _build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ("tb_from_ijk", "tb_from_leaves", "tb_refine", "tb_coarsen", "tb_box_dilate",
                 "tb_chain", "tb_multi", "tb_refine_masked", "tb_batch_free", "tb_batch_get_view", "tb_validate",
                 "tb_last_error"):
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_build_targets_sm103a_only():
    from sparse_voxel_grid_leaf_gb300 import _build
    assert _build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_host_side_argument_errors(lib):
    lib.tb_last_error.restype = ctypes.c_char_p
    lib.tb_status_string.restype = ctypes.c_char_p
    lib.tb_version.restype = ctypes.c_int32
    assert lib.tb_version() >= 100
    assert lib.tb_status_string(4) == b"TB_ERR_COORD_OVERFLOW"
    # out == NULL is rejected before any CUDA call
    st = lib.tb_from_ijk(None, None, ctypes.c_int32(1), ctypes.c_int64(0), None, None, None)
    assert st == 1
    assert b"bad pointer" in lib.tb_last_error()
    out = ctypes.c_void_p(123)
    st = lib.tb_chain(None, None, ctypes.c_int32(-1), None, None, ctypes.byref(out))
    assert st == 1 and out.value is None
    out = ctypes.c_void_p(123)
    st = lib.tb_refine_masked(None, None, ctypes.c_int32(2), None, None, ctypes.byref(out))
    assert st == 1 and out.value is None
    assert b"batch is NULL" in lib.tb_last_error()
    st = lib.tb_batch_export_many(None, ctypes.c_int32(2), None, None, None, None, None)
    assert st == 1 and b"bad batch list" in lib.tb_last_error()
    st = lib.tb_selftest_wait(ctypes.c_int32(0), ctypes.c_int32(0), None)  # a bad limit, before any CUDA call
    assert st == 1
    st = lib.tb_batch_get_view(None, None)
    assert st == 1
    assert lib.tb_batch_free(None, None) == 0


def test_static_refine_host_checks(lib):
    """tb_refine_static answers before any launch: an input too large for its
    static scratch array, and a host-resident leaf_offsets array."""
    import numpy as np
    lib.tb_last_error.restype = ctypes.c_char_p
    out = (ctypes.c_byte * 256)()   # a zeroed tb_out_buffers (152 bytes)
    offs = np.array([0, 0], np.int64)
    st = lib.tb_refine_static(None, None, ctypes.c_void_p(offs.ctypes.data), ctypes.c_int32(1), ctypes.c_int64(0),
                              ctypes.byref(out), None, None)
    assert st == 1 and b"device memory" in lib.tb_last_error()
    st = lib.tb_refine_static(ctypes.c_void_p(64), ctypes.c_void_p(64), ctypes.c_void_p(offs.ctypes.data),
                              ctypes.c_int32(1), ctypes.c_int64(80660), ctypes.byref(out), None, None)
    assert st == 7 and b"32 MiB" in lib.tb_last_error()


def test_launch_mode_switch(lib):
    # process-wide, host only: returns the previous mode, rejects others
    lib.tb_set_launch_mode.restype = ctypes.c_int32
    prev = lib.tb_set_launch_mode(ctypes.c_int32(2))
    try:
        assert prev in (0, 1, 2)
        assert lib.tb_set_launch_mode(ctypes.c_int32(1)) == 2
        assert lib.tb_set_launch_mode(ctypes.c_int32(3)) == -1
        assert lib.tb_set_launch_mode(ctypes.c_int32(-1)) == -1
        assert lib.tb_set_launch_mode(ctypes.c_int32(0)) == 1
    finally:
        lib.tb_set_launch_mode(ctypes.c_int32(prev))


def test_stride1_box_rule():
    """The K -> box rule, written once in the library: odd K symmetric, even K
    with the extra offset on the positive side, transpose mirrored."""
    import sparse_voxel_grid_leaf_gb300 as tb
    for K, lo, hi in ((1, 0, 0), (2, 0, 1), (3, -1, 1), (4, -1, 2), (5, -2, 2), (15, -7, 7)):
        assert tb.stride1_box(K) == ((lo,) * 3, (hi,) * 3)
        assert tb.stride1_box(K, True) == ((-hi,) * 3, (-lo,) * 3)
    for K in (0, 16, -3):
        with pytest.raises(tb.TBError):
            tb.stride1_box(K)


def test_kmap_mode_switch(lib):
    lib.tb_set_kmap_mode.restype = ctypes.c_int32
    prev = lib.tb_set_kmap_mode(ctypes.c_int32(4))
    try:
        assert prev in range(5)
        assert lib.tb_set_kmap_mode(ctypes.c_int32(1)) == 4
        assert lib.tb_set_kmap_mode(ctypes.c_int32(5)) == -1
        assert lib.tb_set_kmap_mode(ctypes.c_int32(-1)) == -1
        assert lib.tb_set_kmap_mode(ctypes.c_int32(0)) == 1
    finally:
        lib.tb_set_kmap_mode(ctypes.c_int32(prev))


def test_python_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import sparse_voxel_grid_leaf_gb300 as tb
    monkeypatch.setattr(tb, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(tb, "_lib", None)
    with pytest.raises(tb.TBError):
        tb.lib()
