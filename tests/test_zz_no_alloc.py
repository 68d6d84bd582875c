"""vbm_build_device_noalloc: the grid builder for callers that cannot allocate
device memory (code inside an application whose device memory belongs to an
allocator it does not own, or code running while another thread captures a
CUDA graph, when cudaMalloc is refused).

The entry point is called through the C ABI (ctypes) with caller-provided
output memory, twice in a row on different inputs, and each grid it returns
must behave exactly like the one vbm_build_device builds from the same input:
same statistics, same decode maps, same filter outputs bit for bit (the
library's tolerance is 0 ULP).  Collected last, so that a run stopping at the
first failure has already run every other test; it passes alone in a fresh
process as well, since its first call performs the one-time set-up.
"""
import ctypes

import numpy as np
import pytest

import sparse_voxel_grid_gb300 as vbm
import synth
from sparse_voxel_grid_gb300 import _lib
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu

MAX_VOXELS = 65536
STATS = ["n_active", "n_leaves", "n_blocks", "block_width", "n_upper", "n_lower", "n_blocks_over_cache",
         "max_span", "device_bytes"]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    gu.require_gpu()


def _noalloc_build(coords_dev, n, log2w, arena, arena_bytes):
    """Returns (status, handle or None, bytes needed)."""
    t = gu.torch()
    lib = _lib.load()
    h = ctypes.c_void_p()
    need = ctypes.c_uint64(0)
    rc = lib.vbm_build_device_noalloc(ctypes.c_void_p(coords_dev.data_ptr()) if n else None, n, log2w, 0,
                                      ctypes.c_void_p(arena.data_ptr()) if arena is not None else None,
                                      arena_bytes, ctypes.byref(need),
                                      ctypes.c_void_p(t.cuda.current_stream().cuda_stream), ctypes.byref(h))
    return rc, (vbm.Grid(h.value) if rc == 0 else None), int(need.value)


def _check_same(grid, ref):
    for k in STATS:
        assert grid.info[k] == ref.info[k], k
    li, vo = gu.decode(grid)
    rli, rvo = gu.decode(ref)
    np.testing.assert_array_equal(li, rli)
    np.testing.assert_array_equal(vo, rvo)
    for C, resolver in ((1, vbm.RESOLVE_BRICK), (3, vbm.RESOLVE_BRICK), (1, vbm.RESOLVE_CACHED)):
        s = gu.to_dev(synth.sidecar_uniform(ref.n, C, seed=7))
        a = gu.box_filter(grid, s, C, resolver, vbm.OUTPUT_STREAMED)
        b = gu.box_filter(ref, s, C, resolver, vbm.OUTPUT_STREAMED)
        np.testing.assert_array_equal(gu.bits(a), gu.bits(b))
    s = gu.to_dev(synth.sidecar_uniform(ref.n, 1, seed=8))
    np.testing.assert_array_equal(gu.bits(gu.cross_filter(grid, s, 1, vbm.RESOLVE_CACHED, vbm.CROSS_LAPLACIAN)),
                                  gu.bits(gu.cross_filter(ref, s, 1, vbm.RESOLVE_CACHED, vbm.CROSS_LAPLACIAN)))


def test_two_calls_in_a_row_match_the_allocating_builder():
    t = gu.torch()
    inputs = [synth.WORKLOADS["T"](), synth.dense_random((30, 25, 40), 0.35, seed=4, origin=(-9, 17, -40))]
    assert all(len(c) <= MAX_VOXELS for c in inputs)
    for log2w, coords in zip((7, 6), inputs):
        cd = t.from_numpy(coords).cuda()
        # size query: no arena
        rc, g, need = _noalloc_build(cd, len(coords), log2w, None, 0)
        assert rc == _lib.header_constants()["VBM_ERR_RANGE"] and g is None and need > 0
        arena = t.empty(need, dtype=t.uint8, device="cuda")
        rc, g, need2 = _noalloc_build(cd, len(coords), log2w, arena, need)
        assert rc == 0, vbm.vbm_last_error()
        assert need2 == need
        ref = vbm.vbm_build_device(cd, log2w)
        _check_same(g, ref)
        g.close()  # frees the handle only; the arena stays the caller's
        del arena


def test_rejects_inputs_over_the_static_maximum():
    t = gu.torch()
    coords = synth.dense_random((41, 41, 41), 1.0, seed=0)  # 68,921 voxels
    assert len(coords) > MAX_VOXELS
    cd = t.from_numpy(coords).cuda()
    rc, g, need = _noalloc_build(cd, len(coords), 7, None, 0)
    assert rc == _lib.header_constants()["VBM_ERR_RANGE"] and g is None
    assert "65536" in vbm.vbm_last_error()


def test_second_call_allocates_no_device_memory():
    """After the first call on the device (which looks up the static array and
    loads the kernels), a call with the same input changes the device's free
    memory by not one byte."""
    t = gu.torch()
    coords = synth.WORKLOADS["T"]()
    cd = t.from_numpy(coords).cuda()
    rc, g, need = _noalloc_build(cd, len(coords), 7, None, 0)
    assert g is None and need > 0
    arenas = [t.empty(need, dtype=t.uint8, device="cuda") for _ in range(2)]
    rc, g1, _ = _noalloc_build(cd, len(coords), 7, arenas[0], need)
    assert rc == 0, vbm.vbm_last_error()
    t.cuda.synchronize()
    free_before, _ = t.cuda.mem_get_info()
    rc, g2, _ = _noalloc_build(cd, len(coords), 7, arenas[1], need)
    t.cuda.synchronize()
    free_after, _ = t.cuda.mem_get_info()
    assert rc == 0, vbm.vbm_last_error()
    assert free_after == free_before, (free_before, free_after)
    ref = vbm.vbm_build_device(cd, 7)
    _check_same(g2, ref)
    _check_same(g1, ref)
    for g_ in (g1, g2, ref):
        g_.close()


def test_empty_input_needs_a_small_arena():
    """n = 0: the size query asks for a non-empty arena (256 bytes), and the
    empty grid built in it filters like any empty grid (row 0 written as +0.0)."""
    t = gu.torch()
    cd = t.zeros((0, 3), dtype=t.int32, device="cuda")
    rc, g, need = _noalloc_build(cd, 0, 7, None, 0)
    assert rc == _lib.header_constants()["VBM_ERR_RANGE"] and g is None and need == 256
    arena = t.empty(need, dtype=t.uint8, device="cuda")
    rc, g, _ = _noalloc_build(cd, 0, 7, arena, need)
    assert rc == 0, vbm.vbm_last_error()
    assert g.n == 0 and g.n_slots == 0 and g.info["on_device"] == 1
    s = t.ones(3, device="cuda")
    out = t.full((3,), 5.0, device="cuda")
    vbm.vbm_box_filter(g, s, 3, out, vbm.RESOLVE_BRICK)
    t.cuda.synchronize()
    assert (out.cpu() == 0).all()
    g.close()
