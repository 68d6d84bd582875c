"""ctypes binding of libvbm.so (include/vbm.h).  Argument marshalling only:
every step of the pipeline runs in the library's CUDA kernels.  There is no
fallback: if libvbm.so is missing, loading fails with an error."""
from __future__ import annotations

import ctypes
import os
import re
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libvbm.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
HEADER = os.path.join(INCLUDE, "vbm.h")
HEADERS = [os.path.join(INCLUDE, f) for f in ("vbm.h", "vbm_probe.h")]


def _header_text() -> str:
    return "\n".join(open(h).read() for h in HEADERS)

_lock = threading.Lock()
_lib = None


class VbmError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"[{code}] {msg}")
        self.code = code


def header_constants() -> dict:
    """#define NAME value pairs of the headers in include/ (integers only)."""
    out = {}
    for m in re.finditer(r"^#define\s+(VBM_\w+)\s+\(?(-?\w+)u?\)?", _header_text(), re.M):
        try:
            out[m.group(1)] = int(m.group(2).rstrip("u"), 0)
        except ValueError:
            pass
    return out


def header_functions() -> list:
    """Names of the functions the headers in include/ declare."""
    return sorted(set(re.findall(r"^(?:int|const char\*)\s+(vbm_\w+)\s*\(", _header_text(), re.M)))


class VbmInfo(ctypes.Structure):
    _fields_ = [
        ("n_active", ctypes.c_uint64),
        ("n_leaves", ctypes.c_uint64),
        ("n_blocks", ctypes.c_uint64),
        ("block_width", ctypes.c_uint32),
        ("log2_block_width", ctypes.c_uint32),
        ("n_upper", ctypes.c_uint32),
        ("n_lower", ctypes.c_uint32),
        ("n_blocks_over_cache", ctypes.c_uint64),
        ("max_span", ctypes.c_uint32),
        ("on_device", ctypes.c_uint32),
        ("device_bytes", ctypes.c_uint64),
    ]


def load(path: str = LIB_PATH):
    """Load libvbm.so (once).  Raises OSError if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise OSError(f"libvbm.so not found at {path}: build it with "
                              "`python -m sparse_voxel_grid_gb300._build`")
            lib = ctypes.CDLL(path)
            p, i32, u32, u64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint32, ctypes.c_uint64
            lib.vbm_last_error.restype = ctypes.c_char_p
            lib.vbm_last_error.argtypes = []
            lib.vbm_build.restype = i32
            lib.vbm_build.argtypes = [p, u64, i32, u32, p, ctypes.POINTER(p)]
            lib.vbm_build_device.restype = i32
            lib.vbm_build_device.argtypes = [p, u64, i32, u32, p, ctypes.POINTER(p)]
            lib.vbm_build_device_noalloc.restype = i32
            lib.vbm_build_device_noalloc.argtypes = [p, u64, i32, u32, p, u64, ctypes.POINTER(u64), p,
                                                     ctypes.POINTER(p)]
            lib.vbm_destroy.restype = i32
            lib.vbm_destroy.argtypes = [p]
            lib.vbm_info.restype = i32
            lib.vbm_info.argtypes = [p, ctypes.POINTER(VbmInfo)]
            lib.vbm_leaf_export.restype = i32
            lib.vbm_leaf_export.argtypes = [p, i32, p, u64]
            lib.vbm_decode.restype = i32
            lib.vbm_decode.argtypes = [p, p, p, p]
            lib.vbm_decode_sweep.restype = i32
            lib.vbm_decode_sweep.argtypes = [p, p, p, p]
            lib.vbm_box_filter.restype = i32
            lib.vbm_box_filter.argtypes = [p, p, i32, p, i32, i32, p]
            lib.vbm_box_filter_batch.restype = i32
            lib.vbm_box_filter_batch.argtypes = [p, i32, p, p, p, i32, p]
            lib.vbm_box_filter_batch_host.restype = i32
            lib.vbm_box_filter_batch_host.argtypes = [p, i32, p, p, p, i32, p]
            lib.vbm_shard_blocks.restype = i32
            lib.vbm_shard_blocks.argtypes = [p, i32, p]
            lib.vbm_shard_halo.restype = i32
            lib.vbm_shard_halo.argtypes = [p, u32, u32, p, u64, ctypes.POINTER(u64)]
            lib.vbm_gather_rows.restype = i32
            lib.vbm_gather_rows.argtypes = [p, i32, p, u64, p, p]
            lib.vbm_scatter_rows.restype = i32
            lib.vbm_scatter_rows.argtypes = [p, i32, p, u64, p, p]
            lib.vbm_box_filter_batch_blocks.restype = i32
            lib.vbm_box_filter_batch_blocks.argtypes = [p, u32, u32, i32, p, p, p, i32, p]
            lib.vbm_cross_filter.restype = i32
            lib.vbm_cross_filter.argtypes = [p, p, i32, p, i32, i32, p]
            lib.vbm_box_taps.restype = i32
            lib.vbm_box_taps.argtypes = [p, p, i32, p]
            lib.vbm_cross_taps.restype = i32
            lib.vbm_cross_taps.argtypes = [p, p, i32, p]
            lib.vbm_weno_filter.restype = i32
            lib.vbm_weno_filter.argtypes = [p, p, ctypes.c_float, p, i32, p]
            lib.vbm_weno_taps.restype = i32
            lib.vbm_weno_taps.argtypes = [p, p, i32, p]
            lib.vbm_probe_launch.restype = i32
            lib.vbm_probe_launch.argtypes = [p, i32, p, p]
            _lib = lib
    return _lib


def check(rc: int) -> None:
    if rc != 0:
        raise VbmError(rc, load().vbm_last_error().decode(errors="replace"))
