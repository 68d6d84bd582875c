"""GB300 (sm_103a) sparse voxel-grid stencils in the style of NanoVDB's
VoxelBlockManager: select-based inverse-map decode, 27-tap box and 7-tap cross
stencil resolution by tree walk or a cached neighbour-leaf table, and fused
gather-and-accumulate filters over C interleaved fp32 sidecar channels.

The compute path is libvbm.so (C ABI, include/vbm.h).  This module is a thin
binding with the same function names: it checks and marshals arguments (torch
CUDA tensors for device memory, torch streams) and calls the library.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import _lib
from ._lib import VbmError, VbmInfo, check, load

_K = _lib.header_constants()
OK = _K["VBM_OK"]
MAX_CACHED_LEAVES = _K["VBM_MAX_CACHED_LEAVES"]
BUILD_DEDUP = _K["VBM_BUILD_DEDUP"]
BUILD_HOST_ONLY = _K["VBM_BUILD_HOST_ONLY"]
RESOLVE_TREEWALK = _K["VBM_RESOLVE_TREEWALK"]
RESOLVE_CACHED = _K["VBM_RESOLVE_CACHED"]
RESOLVE_BRICK = _K["VBM_RESOLVE_BRICK"]
OUTPUT_STREAMED = _K["VBM_OUTPUT_STREAMED"]
OUTPUT_MATERIALISED = _K["VBM_OUTPUT_MATERIALISED"]
CROSS_LAPLACIAN = _K["VBM_CROSS_LAPLACIAN"]
CROSS_SUM = _K["VBM_CROSS_SUM"]
PROBE_EMPTY = _K["VBM_PROBE_EMPTY"]
PROBE_METADATA = _K["VBM_PROBE_METADATA"]
PROBE_CHAIN = _K["VBM_PROBE_CHAIN"]
EXPORT = {
    "leaf_mask": (_K["VBM_EXPORT_LEAF_MASK"], np.uint64, 8),
    "leaf_prefix": (_K["VBM_EXPORT_LEAF_PREFIX"], np.uint64, 1),
    "leaf_first": (_K["VBM_EXPORT_LEAF_FIRST"], np.uint32, 1),
    "leaf_origin": (_K["VBM_EXPORT_LEAF_ORIGIN"], np.int32, 3),
    "block_first_leaf": (_K["VBM_EXPORT_BLOCK_FIRST_LEAF"], np.uint32, 1),
    "block_jump": (_K["VBM_EXPORT_BLOCK_JUMP"], np.uint64, None),
    "leaf_neighbours": (_K["VBM_EXPORT_LEAF_NEIGHBOURS"], np.uint32, 32),
}
BOX_TAPS = 27
CROSS_TAPS = 7
WENO_TAPS = 19
SENTINEL_LEAF = 0xFFFFFFFF
SENTINEL_OFFSET = 0xFFFF

__all__ = [
    "Grid", "VbmError", "vbm_build", "vbm_build_device", "vbm_destroy", "vbm_info", "vbm_leaf_export", "vbm_decode",
    "vbm_decode_sweep", "vbm_box_filter", "vbm_box_filter_batch", "vbm_box_filter_batch_host", "vbm_cross_filter", "vbm_weno_filter", "vbm_box_taps", "vbm_cross_taps",
    "vbm_weno_taps", "vbm_last_error", "vbm_probe_launch",
]


class Grid:
    """Owns a vbm_grid handle; destroyed with vbm_destroy on close()/GC."""

    def __init__(self, handle: int):
        self._h = ctypes.c_void_p(handle)
        self._info = None

    @property
    def handle(self) -> ctypes.c_void_p:
        if not self._h:
            raise VbmError(_K["VBM_ERR_INVALID"], "grid already destroyed")
        return self._h

    def close(self) -> None:
        if getattr(self, "_h", None):
            check(load().vbm_destroy(self._h))
            self._h = ctypes.c_void_p(None)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def info(self) -> dict:
        if self._info is None:
            self._info = vbm_info(self)
        return self._info

    @property
    def n(self) -> int:
        return self.info["n_active"]

    @property
    def log2w(self) -> int:
        return self.info["log2_block_width"]

    @property
    def n_slots(self) -> int:
        return self.info["n_blocks"] * self.info["block_width"]


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _dev_ptr(t, dtype, numel: int, name: str) -> ctypes.c_void_p:
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements, got {t.numel()}")
    return ctypes.c_void_p(t.data_ptr())


def vbm_last_error() -> str:
    return load().vbm_last_error().decode(errors="replace")


def vbm_build(coords, log2_block_width: int = 7, flags: int = 0, stream=None) -> Grid:
    """Build a grid from an (N,3) int32 host array of active coordinates."""
    c = np.ascontiguousarray(np.asarray(coords, dtype=np.int32).reshape(-1, 3))
    h = ctypes.c_void_p()
    s = ctypes.c_void_p(None) if (flags & BUILD_HOST_ONLY) else _stream_handle(stream)
    check(load().vbm_build(c.ctypes.data if len(c) else None, len(c), int(log2_block_width), int(flags), s,
                           ctypes.byref(h)))
    return Grid(h.value)


def vbm_build_device(coords, log2_block_width: int = 7, flags: int = 0, stream=None) -> Grid:
    """Build a grid on the GPU from an (N,3) int32 CUDA tensor of coordinates."""
    import torch
    if not isinstance(coords, torch.Tensor) or not coords.is_cuda or coords.dtype != torch.int32:
        raise TypeError("coords must be an int32 CUDA tensor")
    c = coords.reshape(-1, 3).contiguous()
    h = ctypes.c_void_p()
    check(load().vbm_build_device(ctypes.c_void_p(c.data_ptr()) if c.numel() else None, c.shape[0],
                                  int(log2_block_width), int(flags), _stream_handle(stream), ctypes.byref(h)))
    return Grid(h.value)


def vbm_destroy(grid: Grid) -> None:
    grid.close()


def vbm_info(grid: Grid) -> dict:
    info = VbmInfo()
    check(load().vbm_info(grid.handle, ctypes.byref(info)))
    return {name: int(getattr(info, name)) for name, _ in VbmInfo._fields_}


def vbm_leaf_export(grid: Grid, what: str) -> np.ndarray:
    """Host copy of one builder array (see EXPORT)."""
    code, dtype, width = EXPORT[what]
    info = grid.info
    if what.startswith("leaf_"):
        shape = (info["n_leaves"], width) if width > 1 else (info["n_leaves"],)
    elif what == "block_jump":
        shape = (info["n_blocks"], info["block_width"] // 64)
    else:
        shape = (info["n_blocks"],)
    out = np.empty(shape, dtype=dtype)
    check(load().vbm_leaf_export(grid.handle, code, out.ctypes.data if out.size else None, out.nbytes))
    return out


def vbm_decode(grid: Grid, leaf_index, voxel_offset, stream=None) -> None:
    """leaf_index: uint32 (as torch.int32) and voxel_offset: uint16 (as
    torch.int16) CUDA tensors of n_blocks*W entries."""
    import torch
    m = grid.n_slots
    check(load().vbm_decode(grid.handle, _dev_ptr(leaf_index, torch.int32, m, "leaf_index"),
                            _dev_ptr(voxel_offset, torch.int16, m, "voxel_offset"), _stream_handle(stream)))


def vbm_decode_sweep(grid: Grid, leaf_index, voxel_offset, stream=None) -> None:
    """The sweep decode (the select decode's predecessor): same arguments and
    the same output bits as vbm_decode."""
    import torch
    m = grid.n_slots
    check(load().vbm_decode_sweep(grid.handle, _dev_ptr(leaf_index, torch.int32, m, "leaf_index"),
                                  _dev_ptr(voxel_offset, torch.int16, m, "voxel_offset"), _stream_handle(stream)))


def vbm_box_filter(grid: Grid, sidecar, C: int, out, resolver: int = RESOLVE_CACHED,
                   output: int = OUTPUT_STREAMED, stream=None) -> None:
    """27-tap box filter of (N+1)*C float32 CUDA tensors (see include/vbm.h)."""
    import torch
    m = (grid.n + 1) * C
    check(load().vbm_box_filter(grid.handle, _dev_ptr(sidecar, torch.float32, m, "sidecar"), int(C),
                                _dev_ptr(out, torch.float32, m, "out"), int(resolver), int(output),
                                _stream_handle(stream)))


def vbm_box_filter_batch(grid: Grid, sidecars, Cs, outs, resolver: int = RESOLVE_BRICK, stream=None) -> None:
    """Box filters of several (N+1)*C float32 CUDA tensors in one call (see
    include/vbm.h): outs[i] = box(sidecars[i]) with Cs[i] channels."""
    import torch
    k = len(sidecars)
    if not (len(Cs) == len(outs) == k):
        raise ValueError("sidecars, Cs and outs must have the same length")
    sc = (ctypes.c_void_p * max(k, 1))()
    ou = (ctypes.c_void_p * max(k, 1))()
    cs = (ctypes.c_int * max(k, 1))()
    for i in range(k):
        m = (grid.n + 1) * int(Cs[i])
        sc[i] = _dev_ptr(sidecars[i], torch.float32, m, "sidecar").value
        ou[i] = _dev_ptr(outs[i], torch.float32, m, "out").value
        cs[i] = int(Cs[i])
    check(load().vbm_box_filter_batch(grid.handle, k, sc, cs, ou, int(resolver), _stream_handle(stream)))


def vbm_cross_filter(grid: Grid, sidecar, C: int, out, resolver: int = RESOLVE_CACHED,
                     op: int = CROSS_LAPLACIAN, stream=None) -> None:
    """7-tap cross consumer (Laplacian or sum) of (N+1)*C float32 CUDA tensors."""
    import torch
    m = (grid.n + 1) * C
    check(load().vbm_cross_filter(grid.handle, _dev_ptr(sidecar, torch.float32, m, "sidecar"), int(C),
                                  _dev_ptr(out, torch.float32, m, "out"), int(resolver), int(op),
                                  _stream_handle(stream)))


def vbm_box_taps(grid: Grid, taps, resolver: int = RESOLVE_CACHED, stream=None) -> None:
    """(N+1)*27 uint32 (as torch.int32) CUDA tensor of raw box taps."""
    import torch
    check(load().vbm_box_taps(grid.handle, _dev_ptr(taps, torch.int32, (grid.n + 1) * BOX_TAPS, "taps"),
                              int(resolver), _stream_handle(stream)))


def vbm_cross_taps(grid: Grid, taps, resolver: int = RESOLVE_CACHED, stream=None) -> None:
    """(N+1)*7 uint32 (as torch.int32) CUDA tensor of raw cross taps."""
    import torch
    check(load().vbm_cross_taps(grid.handle, _dev_ptr(taps, torch.int32, (grid.n + 1) * CROSS_TAPS, "taps"),
                                int(resolver), _stream_handle(stream)))


def vbm_weno_filter(grid: Grid, phi, out, iso: float = 0.0, resolver: int = RESOLVE_CACHED, stream=None) -> None:
    """19-tap WENO consumer (Godunov squared gradient norm) of an N+1 float32
    CUDA tensor phi (row 0 the background value) into out (N+1 float32)."""
    import torch
    m = grid.n + 1
    check(load().vbm_weno_filter(grid.handle, _dev_ptr(phi, torch.float32, m, "phi"), float(iso),
                                 _dev_ptr(out, torch.float32, m, "out"), int(resolver), _stream_handle(stream)))


def vbm_weno_taps(grid: Grid, taps, resolver: int = RESOLVE_CACHED, stream=None) -> None:
    """(N+1)*19 uint32 (as torch.int32) CUDA tensor of raw WENO taps."""
    import torch
    check(load().vbm_weno_taps(grid.handle, _dev_ptr(taps, torch.int32, (grid.n + 1) * WENO_TAPS, "taps"),
                               int(resolver), _stream_handle(stream)))


def vbm_probe_launch(grid: Grid, kind: int, sidecar=None, stream=None) -> None:
    """A measurement probe with the grid's filter launch shape (include/vbm_probe.h):
    PROBE_EMPTY, PROBE_METADATA, or PROBE_CHAIN (reads `sidecar`, N+1 float32)."""
    import torch
    p = _dev_ptr(sidecar, torch.float32, grid.n + 1, "sidecar") if sidecar is not None else None
    check(load().vbm_probe_launch(grid.handle, int(kind), p, _stream_handle(stream)))


def _host_ptr(a, numel: int, name: str) -> int:
    """Address of a contiguous float32 host array (numpy or CPU torch tensor)."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            if a.is_cuda or a.dtype != torch.float32 or not a.is_contiguous():
                raise TypeError(f"{name} must be a contiguous float32 CPU tensor")
            if a.numel() != numel:
                raise ValueError(f"{name} must have {numel} elements, got {a.numel()}")
            return a.data_ptr()
    except ImportError:
        pass
    if not isinstance(a, np.ndarray) or a.dtype != np.float32 or not a.flags["C_CONTIGUOUS"]:
        raise TypeError(f"{name} must be a contiguous float32 host array")
    if a.size != numel:
        raise ValueError(f"{name} must have {numel} elements, got {a.size}")
    return a.ctypes.data


def vbm_box_filter_batch_host(grid: Grid, host_sidecars, Cs, host_outs, resolver: int = RESOLVE_BRICK,
                              stream=None) -> None:
    """vbm_box_filter_batch on host-resident (N+1)*C float32 arrays (numpy or
    CPU torch tensors; pinned memory gives overlapped copies).  Only enqueues:
    the outputs are ready once `stream` is synchronised (see include/vbm.h)."""
    k = len(host_sidecars)
    if not (len(Cs) == len(host_outs) == k):
        raise ValueError("host_sidecars, Cs and host_outs must have the same length")
    sc = (ctypes.c_void_p * max(k, 1))()
    ou = (ctypes.c_void_p * max(k, 1))()
    cs = (ctypes.c_int * max(k, 1))()
    for i in range(k):
        m = (grid.n + 1) * int(Cs[i])
        sc[i] = _host_ptr(host_sidecars[i], m, "host sidecar")
        ou[i] = _host_ptr(host_outs[i], m, "host output")
        cs[i] = int(Cs[i])
    check(load().vbm_box_filter_batch_host(grid.handle, k, sc, cs, ou, int(resolver), _stream_handle(stream)))
