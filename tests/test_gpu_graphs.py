"""Every compute call only enqueues kernels on the given stream: captured into
a CUDA graph and replayed, each gives the bits of a direct call, and two
streams may run calls on one grid at the same time."""
import numpy as np
import pytest

import sparse_voxel_grid_gb300 as vbm
import synth
from tests import gpu_util as gu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    gu.require_gpu()


@pytest.mark.parametrize("log2w", [7, 9])
def test_graph_capture_and_replay(log2w):
    t = gu.torch()
    coords = synth.WORKLOADS["T"]()
    g = vbm.vbm_build(coords, log2w)
    n = g.n
    side = {C: t.from_numpy(synth.sidecar_uniform(n, C, seed=C)).cuda() for C in (1, 3, 16)}
    direct = {}
    for C in (1, 3, 16):
        o = t.empty_like(side[C])
        vbm.vbm_box_filter(g, side[C], C, o, vbm.RESOLVE_BRICK)
        direct[("box", C)] = o
    lap = t.empty_like(side[1])
    vbm.vbm_cross_filter(g, side[1], 1, lap, vbm.RESOLVE_CACHED, vbm.CROSS_LAPLACIAN)
    weno = t.empty_like(side[1])
    vbm.vbm_weno_filter(g, side[1], weno, 0.0, vbm.RESOLVE_BRICK)
    li = t.empty(g.n_slots, dtype=t.int32, device="cuda")
    vo = t.empty(g.n_slots, dtype=t.int16, device="cuda")
    vbm.vbm_decode(g, li, vo)
    t.cuda.synchronize()
    bouts = {C: t.full_like(side[C], float("nan")) for C in (1, 3, 16)}

    outs = {C: t.full_like(side[C], float("nan")) for C in (1, 3, 16)}
    glap, gweno = t.full_like(lap, float("nan")), t.full_like(weno, float("nan"))
    gli, gvo = t.zeros_like(li), t.zeros_like(vo)
    s = t.cuda.Stream()
    graph = t.cuda.CUDAGraph()
    with t.cuda.stream(s):
        with t.cuda.graph(graph, stream=s):
            for C in (1, 3, 16):
                vbm.vbm_box_filter(g, side[C], C, outs[C], vbm.RESOLVE_BRICK, stream=s)
            vbm.vbm_cross_filter(g, side[1], 1, glap, vbm.RESOLVE_CACHED, vbm.CROSS_LAPLACIAN, stream=s)
            vbm.vbm_weno_filter(g, side[1], gweno, 0.0, vbm.RESOLVE_BRICK, stream=s)
            vbm.vbm_decode(g, gli, gvo, stream=s)
            vbm.vbm_box_filter_batch(g, [side[C] for C in (1, 3, 16)], [1, 3, 16], [bouts[C] for C in (1, 3, 16)],
                                     vbm.RESOLVE_BRICK, stream=s)
    for _ in range(2):
        graph.replay()
    t.cuda.synchronize()
    for C in (1, 3, 16):
        np.testing.assert_array_equal(gu.bits(outs[C].cpu().numpy()), gu.bits(direct[("box", C)].cpu().numpy()))
    np.testing.assert_array_equal(gu.bits(glap.cpu().numpy()), gu.bits(lap.cpu().numpy()))
    np.testing.assert_array_equal(gu.bits(gweno.cpu().numpy()), gu.bits(weno.cpu().numpy()))
    assert t.equal(gli, li) and t.equal(gvo, vo)
    for C in (1, 3, 16):
        np.testing.assert_array_equal(gu.bits(bouts[C].cpu().numpy()), gu.bits(direct[("box", C)].cpu().numpy()))


def test_two_streams_on_one_grid():
    t = gu.torch()
    coords = synth.WORKLOADS["S185"]()
    g = vbm.vbm_build(coords, 9)
    a = t.from_numpy(synth.sidecar_uniform(g.n, 8, seed=1)).cuda()
    b = t.from_numpy(synth.sidecar_uniform(g.n, 8, seed=2)).cuda()
    ra, rb = t.empty_like(a), t.empty_like(b)
    vbm.vbm_box_filter(g, a, 8, ra, vbm.RESOLVE_BRICK)
    vbm.vbm_box_filter(g, b, 8, rb, vbm.RESOLVE_BRICK)
    t.cuda.synchronize()
    s1, s2 = t.cuda.Stream(), t.cuda.Stream()
    oa, ob = t.full_like(a, float("nan")), t.full_like(b, float("nan"))
    for _ in range(3):
        vbm.vbm_box_filter(g, a, 8, oa, vbm.RESOLVE_BRICK, stream=s1)
        vbm.vbm_box_filter(g, b, 8, ob, vbm.RESOLVE_BRICK, stream=s2)
    t.cuda.synchronize()
    assert t.equal(oa.view(t.int32), ra.view(t.int32)) and t.equal(ob.view(t.int32), rb.view(t.int32))


def test_graph_capture_of_the_shard_calls():
    """The block-range filter and the row gather/scatter are plain enqueues
    too: a captured pack -> place -> filter of two block ranges replays to the
    bits of the whole-grid call."""
    import ctypes
    t = gu.torch()
    g = vbm.vbm_build(synth.WORKLOADS["T"](), 7)
    n, C = g.n, 8
    lib = vbm.load()
    src = t.from_numpy(synth.sidecar_uniform(n, C, seed=9)).cuda()
    want = t.empty_like(src)
    vbm.vbm_box_filter(g, src, C, want, vbm.RESOLVE_BRICK)
    rows = t.arange(1, n + 1, dtype=t.int32, device="cuda")  # every row: packed, then placed back
    packed = t.empty(n * C, device="cuda")
    side = t.full_like(src, float("nan"))
    side[:C] = 0.0
    out = t.full_like(src, float("nan"))
    nb = g.info["n_blocks"]
    t.cuda.synchronize()
    P = ctypes.c_void_p
    s = t.cuda.Stream()
    graph = t.cuda.CUDAGraph()
    with t.cuda.stream(s):
        with t.cuda.graph(graph, stream=s):
            h = P(s.cuda_stream)
            assert lib.vbm_gather_rows(P(src.data_ptr()), C, P(rows.data_ptr()), n, P(packed.data_ptr()), h) == 0
            assert lib.vbm_scatter_rows(P(packed.data_ptr()), C, P(rows.data_ptr()), n, P(side.data_ptr()), h) == 0
            for b0, b1 in ((0, nb // 2), (nb // 2, nb)):
                sc = (ctypes.c_void_p * 1)(side.data_ptr())
                ou = (ctypes.c_void_p * 1)(out.data_ptr())
                cs = (ctypes.c_int * 1)(C)
                assert lib.vbm_box_filter_batch_blocks(g.handle, b0, b1, 1, sc, cs, ou, vbm.RESOLVE_BRICK, h) == 0
    for _ in range(2):
        graph.replay()
    t.cuda.synchronize()
    np.testing.assert_array_equal(gu.bits(out.cpu().numpy()), gu.bits(want.cpu().numpy()))
