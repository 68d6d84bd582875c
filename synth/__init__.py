"""Seeded synthetic inputs for the sparse voxel-grid stencil pipeline.

Shared by the CPU oracle's tests and by the CUDA path's tests and benchmark.
It makes inputs only -- active-voxel coordinate sets and sidecar values -- and
holds none of the pipeline's arithmetic (no tree order, indexing or stencil).

The workloads mirror the ones the pages measure (OpenVDB PR #2263,
"Measurements": a sparse sphere shell of about 1.29M active voxels in 9140
leaves; PR #2258, "A/B - decode", a real VDB data set that is not available
here) with seeded stand-ins: see ``WORKLOADS``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB_PATH = os.path.join(_HERE, "_libsynth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile gen.c into _libsynth.so (plain C, no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-std=c11",
                        _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            i64, u64, i32, dbl, ptr = ctypes.c_int64, ctypes.c_uint64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
            lib.synth_hash64.restype = u64
            lib.synth_hash64.argtypes = [u64, u64]
            lib.synth_sidecar_uniform.restype = None
            lib.synth_sidecar_uniform.argtypes = [u64, i64, i32, ptr]
            lib.synth_sidecar_normal.restype = None
            lib.synth_sidecar_normal.argtypes = [u64, i64, i32, ptr]
            lib.synth_shell.restype = i64
            lib.synth_shell.argtypes = [dbl, dbl, ptr, i64]
            lib.synth_bricks.restype = i64
            lib.synth_bricks.argtypes = [i32, dbl, dbl, dbl, u64, ptr, i64]
            lib.synth_fog_mask.restype = i64
            lib.synth_fog_mask.argtypes = [i32, u64, dbl, ptr]
            lib.synth_mask_coords.restype = i64
            lib.synth_mask_coords.argtypes = [ptr, i32, ptr, i64]
            lib.synth_scatter.restype = i64
            lib.synth_scatter.argtypes = [i32, i64, i32, u64, ptr, i64]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def hash64(seed: int, k: int) -> int:
    return int(_load().synth_hash64(seed, k))


def _two_pass(fn, *args) -> np.ndarray:
    n = fn(*args, None, 0)
    out = np.empty((max(n, 0), 3), dtype=np.int32)
    if n > 0:
        m = fn(*args, _ptr(out), n)
        assert m == n
    return out


def shell(r_in: float, r_out: float) -> np.ndarray:
    """Integer points p with r_in <= |p| <= r_out, as an (N,3) int32 array."""
    return _two_pass(_load().synth_shell, float(r_in), float(r_out))


def bricks(dim_b: int = 64, p_on: float = 0.3, rho_lo: float = 0.01, rho_hi: float = 1.0,
           seed: int = 0) -> np.ndarray:
    """Random 8^3 bricks on [0, 8*dim_b)^3 (see gen.c), (N,3) int32."""
    return _two_pass(_load().synth_bricks, int(dim_b), float(p_on), float(rho_lo), float(rho_hi), int(seed))


def fog(dim: int = 512, seed: int = 0, threshold: float = 0.55) -> np.ndarray:
    """Voxels of [0,dim)^3 where 4-octave value noise exceeds `threshold`."""
    lib = _load()
    mask = np.empty(dim * dim * dim, dtype=np.uint8)
    n = lib.synth_fog_mask(int(dim), int(seed), float(threshold), _ptr(mask))
    if n < 0:
        raise ValueError("fog: dim must be a positive multiple of 64")
    out = np.empty((n, 3), dtype=np.int32)
    m = lib.synth_mask_coords(_ptr(mask), int(dim), _ptr(out), n)
    assert m == n
    return out


def scatter(side: int, count: int, origin: int = 0, seed: int = 0) -> np.ndarray:
    """`count` points, one per 8-aligned brick, bricks in raster order on a
    side^3 cube of bricks starting at `origin` (see gen.c)."""
    return _two_pass(_load().synth_scatter, int(side), int(count), int(origin), int(seed))


def dense_random(shape, density: float, seed: int = 0, origin=(0, 0, 0)) -> np.ndarray:
    """Points of a box of `shape` cells at `origin`, each on with prob `density`."""
    sx, sy, sz = shape
    n = sx * sy * sz
    keys = np.arange(n, dtype=np.uint64)
    lib = _load()
    u = np.fromiter((lib.synth_hash64(seed ^ 0x64656E7365, int(k)) >> 11 for k in keys), dtype=np.uint64, count=n)
    on = (u.astype(np.float64) * (1.0 / 9007199254740992.0)) < density
    idx = np.nonzero(on.reshape(sx, sy, sz))
    pts = np.stack(idx, axis=1).astype(np.int64) + np.asarray(origin, dtype=np.int64)
    return pts.astype(np.int32)


def sidecar_uniform(n: int, C: int, seed: int = 0) -> np.ndarray:
    """(n+1)*C float32 in U[-1,1), row 0 zero; value of (row r, channel c) keyed
    by r*C+c."""
    out = np.empty((n + 1) * C, dtype=np.float32)
    _load().synth_sidecar_uniform(int(seed), int(n), int(C), _ptr(out))
    return out


def sidecar_normal(n: int, C: int, seed: int = 0) -> np.ndarray:
    """(n+1)*C float32 N(0,1) (Box-Muller), row 0 zero."""
    out = np.empty((n + 1) * C, dtype=np.float32)
    _load().synth_sidecar_normal(int(seed), int(n), int(C), _ptr(out))
    return out


# Named workloads: coordinate recipe and the sidecar recipe used with it.
#   T    tiny shell, 11.5 <= |p| <= 13.5, sidecar U[-1,1) seed 0, C=1, W=128
#   S185 shell radius 185, thickness 3: 183.5 <= |p| <= 186.5 (~1.29M voxels)
#   S160 the shell matching the pages' counts: 158 <= |p| <= 162
#        (1,288,594 voxels in 9,140 leaves, occupancy 141/512)
#   D    decode grid: 64^3 bricks of 8^3 on [0,512)^3, p_on 0.3, rho U[0.01,1)
#   F    fog: 512^3 four-octave value noise > 0.55, sidecar N(0,1) C=8, W=256
WORKLOADS = {
    "T": lambda: shell(11.5, 13.5),
    "S185": lambda: shell(183.5, 186.5),
    "S160": lambda: shell(158.0, 162.0),
    "D": lambda: bricks(64, 0.3, 0.01, 1.0, 0),
    "F": lambda: fog(512, 0, 0.55),
}
