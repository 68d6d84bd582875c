"""Helpers for the GPU parity tests: run the library's calls through the
Python binding (which calls the C ABI) and bring results back as numpy."""
from __future__ import annotations

import numpy as np

import sparse_voxel_grid_gb300 as vbm


def torch():
    import torch as t
    return t


def require_gpu():
    import pytest
    t = torch()
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    vbm.load()


def to_dev(a: np.ndarray):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(a)).cuda()


def decode(g, method="select"):
    """Decode maps as (uint32, uint16) host arrays.  The buffers start filled
    with values no decode writes, so a slot left unwritten shows up."""
    t = torch()
    m = g.n_slots
    li = t.full((m,), 0x5A5A5A5A, dtype=t.int32, device="cuda")
    vo = t.full((m,), 0x5555, dtype=t.int16, device="cuda")
    {"select": vbm.vbm_decode, "sweep": vbm.vbm_decode_sweep}[method](g, li, vo)
    t.cuda.synchronize()
    return li.cpu().numpy().view(np.uint32), vo.cpu().numpy().view(np.uint16)


def box_filter(g, sidecar_dev, C, resolver, output):
    t = torch()
    out = t.full(((g.n + 1) * C,), float("nan"), dtype=t.float32, device="cuda")
    vbm.vbm_box_filter(g, sidecar_dev, C, out, resolver, output)
    t.cuda.synchronize()
    return out.cpu().numpy()


def cross_filter(g, sidecar_dev, C, resolver, op):
    t = torch()
    out = t.full(((g.n + 1) * C,), float("nan"), dtype=t.float32, device="cuda")
    vbm.vbm_cross_filter(g, sidecar_dev, C, out, resolver, op)
    t.cuda.synchronize()
    return out.cpu().numpy()


def weno_filter(g, phi_dev, resolver, iso=0.0):
    t = torch()
    out = t.full((g.n + 1,), float("nan"), dtype=t.float32, device="cuda")
    vbm.vbm_weno_filter(g, phi_dev, out, iso, resolver)
    t.cuda.synchronize()
    return out.cpu().numpy()


def taps(g, shape, resolver):
    t = torch()
    out = t.full(((g.n + 1) * shape,), -1, dtype=t.int32, device="cuda")
    {27: vbm.vbm_box_taps, 7: vbm.vbm_cross_taps, 19: vbm.vbm_weno_taps}[shape](g, out, resolver)
    t.cuda.synchronize()
    return out.cpu().numpy().view(np.uint32).reshape(-1, shape)


def bits(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float32).view(np.uint32)
