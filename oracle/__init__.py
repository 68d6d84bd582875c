"""CPU oracle for the sparse voxel-grid stencil pipeline.

TEST INFRASTRUCTURE ONLY.  A plain, slow, obviously correct C++ restatement
(oracle.cpp) of what the pipeline computes.  Only the tests, the smoke check and
the benchmark's CPU-baseline leg may import this package; the product library
never does, and the two share no code.  See oracle.cpp for the readings of the
pages it implements.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_LIB_PATH = os.path.join(_HERE, "_liboracle.so")
_lock = threading.Lock()
_lib = None

SENTINEL_LEAF = 0xFFFFFFFF
SENTINEL_OFFSET = 0xFFFF
CROSS_TAPS = (4, 10, 12, 13, 14, 16, 22)


def build(force: bool = False) -> str:
    """Compile oracle.cpp (no FMA contraction, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["g++", "-std=c++20", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                        _SRC, "-o", tmp], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            p, i64, i32, u32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int32
            lib.oracle_create.restype = p
            lib.oracle_create.argtypes = [p, i64, ctypes.POINTER(ctypes.c_int)]
            lib.oracle_free.restype = None
            lib.oracle_free.argtypes = [p]
            lib.oracle_count.restype = i64
            lib.oracle_count.argtypes = [p]
            lib.oracle_coords.restype = None
            lib.oracle_coords.argtypes = [p, p]
            lib.oracle_index.restype = i64
            lib.oracle_index.argtypes = [p, u32, u32, u32]
            lib.oracle_leaves.restype = i64
            lib.oracle_leaves.argtypes = [p, p, p]
            lib.oracle_decode.restype = None
            lib.oracle_decode.argtypes = [p, i32, p, p]
            lib.oracle_blocks.restype = None
            lib.oracle_blocks.argtypes = [p, i32, p, p]
            lib.oracle_taps.restype = i32
            lib.oracle_taps.argtypes = [p, i32, p, i64, p]
            lib.oracle_box_filter.restype = None
            lib.oracle_box_filter.argtypes = [p, p, i32, p, i64, p]
            lib.oracle_cross_filter.restype = i32
            lib.oracle_cross_filter.argtypes = [p, p, i32, i32, p, i64, p]
            lib.oracle_weno_filter.restype = None
            lib.oracle_weno_filter.argtypes = [p, p, ctypes.c_float, p, i64, p]
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


class OracleGrid:
    """Active voxels in tree order; index i (1..N) is the i-th voxel."""

    def __init__(self, coords: np.ndarray):
        lib = _load()
        c = np.ascontiguousarray(coords, dtype=np.int32).reshape(-1, 3)
        st = ctypes.c_int(0)
        h = lib.oracle_create(_ptr(c), len(c), ctypes.byref(st))
        if not h:
            raise ValueError("oracle: duplicate coordinates")
        self._h = h
        self._lib = lib
        self.n = int(lib.oracle_count(h))

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._lib.oracle_free(h)
            self._h = None

    def coords(self) -> np.ndarray:
        """(N,3) int32; row i-1 holds the coordinate of index i."""
        out = np.empty((self.n, 3), dtype=np.int32)
        self._lib.oracle_coords(self._h, _ptr(out))
        return out

    def index(self, x: int, y: int, z: int) -> int:
        return int(self._lib.oracle_index(self._h, x, y, z))

    def leaves(self):
        """(leaf_of[N+1] uint32, origins[nLeaves,3] int32)."""
        leaf_of = np.empty(self.n + 1, dtype=np.uint32)
        origins = np.empty((max(self.n, 1), 3), dtype=np.int32)
        nl = self._lib.oracle_leaves(self._h, _ptr(leaf_of), _ptr(origins))
        return leaf_of, origins[:nl].copy()

    def n_blocks(self, log2w: int) -> int:
        W = 1 << log2w
        return (self.n + W - 1) // W

    def decode(self, log2w: int):
        """(leaf_index uint32[nBlocks*W], voxel_offset uint16[nBlocks*W])."""
        m = self.n_blocks(log2w) << log2w
        li = np.empty(m, dtype=np.uint32)
        vo = np.empty(m, dtype=np.uint16)
        self._lib.oracle_decode(self._h, log2w, _ptr(li), _ptr(vo))
        return li, vo

    def blocks(self, log2w: int):
        """(firstLeafID uint32[nBlocks], jumpMap uint64[nBlocks, W/64])."""
        nb = self.n_blocks(log2w)
        words = (1 << log2w) // 64
        fl = np.empty(nb, dtype=np.uint32)
        jm = np.empty((nb, words), dtype=np.uint64)
        self._lib.oracle_blocks(self._h, log2w, _ptr(fl), _ptr(jm))
        return fl, jm

    @staticmethod
    def _which(which):
        if which is None:
            return None, 0
        w = np.ascontiguousarray(which, dtype=np.int64)
        return w, len(w)

    def taps(self, shape: int = 27, which=None) -> np.ndarray:
        w, m = self._which(which)
        rows = m if w is not None else self.n + 1
        out = np.empty((rows, shape), dtype=np.uint32)
        rc = self._lib.oracle_taps(self._h, shape, _ptr(w), m, _ptr(out))
        if rc:
            raise ValueError("oracle: shape must be 27, 19 or 7")
        return out

    def box_filter(self, sidecar: np.ndarray, C: int, which=None) -> np.ndarray:
        s = np.ascontiguousarray(sidecar, dtype=np.float32)
        assert s.size == (self.n + 1) * C
        w, m = self._which(which)
        rows = m if w is not None else self.n + 1
        out = np.empty(rows * C, dtype=np.float32)
        self._lib.oracle_box_filter(self._h, _ptr(s), C, _ptr(w), m, _ptr(out))
        return out

    def cross_filter(self, sidecar: np.ndarray, C: int, op: int = 0, which=None) -> np.ndarray:
        s = np.ascontiguousarray(sidecar, dtype=np.float32)
        assert s.size == (self.n + 1) * C
        w, m = self._which(which)
        rows = m if w is not None else self.n + 1
        out = np.empty(rows * C, dtype=np.float32)
        rc = self._lib.oracle_cross_filter(self._h, _ptr(s), C, op, _ptr(w), m, _ptr(out))
        if rc:
            raise ValueError("oracle: op must be 0 (Laplacian) or 1 (7-tap sum)")
        return out

    def weno_filter(self, phi: np.ndarray, iso: float = 0.0, which=None) -> np.ndarray:
        """19-tap WENO consumer: Godunov squared gradient norm of phi (N+1
        float32 rows, row 0 the background) at each row."""
        s = np.ascontiguousarray(phi, dtype=np.float32)
        assert s.size == self.n + 1
        w, m = self._which(which)
        rows = m if w is not None else self.n + 1
        out = np.empty(rows, dtype=np.float32)
        self._lib.oracle_weno_filter(self._h, _ptr(s), float(iso), _ptr(w), m, _ptr(out))
        return out
