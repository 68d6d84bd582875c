"""The C ABI: libvbm.so loads, exports every function include/vbm.h declares,
and rejects bad arguments with status codes before touching the GPU."""
import ctypes

import numpy as np
import pytest

import sparse_voxel_grid_gb300 as vbm
from sparse_voxel_grid_gb300 import _lib


def test_library_exports_every_declared_function():
    lib = _lib.load()
    names = _lib.header_functions()
    assert {"vbm_build", "vbm_decode", "vbm_box_filter", "vbm_cross_filter"} <= set(names)
    for name in names:
        assert hasattr(lib, name), name


def test_header_constants():
    k = _lib.header_constants()
    assert k["VBM_OK"] == 0
    assert k["VBM_MAX_CACHED_LEAVES"] == 16
    codes = [v for n, v in k.items() if n.startswith("VBM_ERR_")]
    assert len(codes) == len(set(codes)) and all(c < 0 for c in codes)


def _raw():
    return _lib.load()


def test_null_and_enum_errors():
    lib = _raw()
    k = _lib.header_constants()
    INVALID, STATE = k["VBM_ERR_INVALID"], k["VBM_ERR_STATE"]
    h = ctypes.c_void_p()
    assert lib.vbm_build(None, 5, 7, 0, None, ctypes.byref(h)) == INVALID
    assert b"coords" in lib.vbm_last_error()
    c = np.zeros((1, 3), dtype=np.int32)
    assert lib.vbm_build(c.ctypes.data, 1, 5, 0, None, ctypes.byref(h)) == INVALID
    assert lib.vbm_build(c.ctypes.data, 1, 10, 0, None, ctypes.byref(h)) == INVALID
    assert lib.vbm_build(c.ctypes.data, 1, 7, 0x100, None, None) == INVALID
    assert lib.vbm_build(c.ctypes.data, 1, 7, 0x100, None, ctypes.byref(h)) == INVALID
    assert lib.vbm_decode(None, None, None, None) == INVALID
    assert lib.vbm_box_filter(None, None, 1, None, 0, 0, None) == INVALID
    assert lib.vbm_cross_filter(None, None, 1, None, 0, 0, None) == INVALID
    assert lib.vbm_box_taps(None, None, 0, None) == INVALID
    assert lib.vbm_cross_taps(None, None, 0, None) == INVALID
    assert lib.vbm_info(None, None) == INVALID
    assert lib.vbm_destroy(None) == 0
    # host-only grid: compute calls refuse with STATE, before any CUDA call
    assert lib.vbm_build(c.ctypes.data, 1, 7, k["VBM_BUILD_HOST_ONLY"], None, ctypes.byref(h)) == 0
    buf = ctypes.c_void_p(256)
    assert lib.vbm_decode(h, buf, buf, None) == STATE
    assert lib.vbm_box_filter(h, buf, 1, buf, 0, 0, None) == STATE
    assert lib.vbm_box_taps(h, buf, 1, None) == STATE
    info = _lib.VbmInfo()
    assert lib.vbm_info(h, ctypes.byref(info)) == 0 and info.on_device == 0 and info.n_active == 1
    # wrong export size
    assert lib.vbm_leaf_export(h, k["VBM_EXPORT_LEAF_FIRST"], ctypes.c_void_p(256), 3) == k["VBM_ERR_RANGE"]
    assert lib.vbm_leaf_export(h, 99, ctypes.c_void_p(256), 4) == INVALID
    assert lib.vbm_destroy(h) == 0


def test_python_binding_errors_carry_text():
    with pytest.raises(vbm.VbmError) as e:
        vbm.vbm_build(np.zeros((1, 3), dtype=np.int32), 4, vbm.BUILD_HOST_ONLY)
    assert "log2_block_width" in str(e.value)
