"""GPU parity on small grids: every output element of the CUDA path (through
the C ABI) against the CPU oracle, bit for bit.

Grids span several VBM blocks and end in a ragged last block; they include
negative coordinates, upper/lower-node boundaries, blocks that overflow the
cached table (one voxel per leaf), and degenerate sizes.
"""
import numpy as np
import pytest

import oracle
import sparse_voxel_grid_gb300 as vbm
import synth
from tests import gpu_util as gu
from tests.test_oracle_pins import GRIDS

pytestmark = pytest.mark.gpu


def _single():
    return np.array([[-3, 7, 12]], dtype=np.int32)


def _exact_blocks(n=256):
    # exactly two blocks of 128 (no partial block) from a dense slab
    c = synth.dense_random((8, 8, 16), 1.0, origin=(0, -4, 0))
    return c[:n]


def _extreme():
    # at the builder's coordinate bound +-2^30, with full stencils around them
    lim = 2 ** 30
    parts = [synth.dense_random((6, 5, 7), 0.6, seed=11, origin=(lim - 5, -lim, lim - 6)),
             synth.dense_random((5, 6, 5), 0.6, seed=12, origin=(-lim, lim - 5, -3)),
             np.array([[lim, lim, lim], [-lim, -lim, -lim], [0, 0, 0]], dtype=np.int32)]
    return np.unique(np.concatenate(parts), axis=0).astype(np.int32)


def _absent_edge_leaves():
    # Taps that cross a leaf's x or y face and its z face at once, into a leaf
    # whose edge-sharing neighbour (the one across the x or y face only) is
    # absent: the tap is active although its z-row's own leaf does not exist.
    rng = np.random.default_rng(21)
    own = np.argwhere(rng.random((8, 8, 8)) < 0.3).astype(np.int32)
    fixed = [(7, 3, 0), (7, 3, 7), (3, 7, 0), (3, 7, 7), (0, 0, 0), (7, 7, 7), (0, 4, 0),  # leaf (0,0,0)
             (8, 3, -1), (8, 3, 8), (9, 2, -3),          # leaves (1,0,-1), (1,0,1)
             (3, 8, -1), (3, 8, 8), (2, 12, 9),          # leaves (0,1,-1), (0,1,1)
             (-1, -1, -1), (-4, -6, -2), (8, 8, 8),      # leaves (-1,-1,-1), (1,1,1)
             (-1, 4, -1), (-1, 4, -8)]                   # leaf (-1,0,-1)
    return np.unique(np.concatenate([own, np.array(fixed, dtype=np.int32)]), axis=0).astype(np.int32)


SMALL = dict(GRIDS)
SMALL.update({
    "extreme": _extreme,
    "scatter": lambda: synth.scatter(side=10, count=700, origin=-37, seed=5),
    "single": _single,
    "exact_blocks": _exact_blocks,
    "exact_plus_one": lambda: _exact_blocks(257),
    "absent_edge_leaves": _absent_edge_leaves,
})

RESOLVERS = [vbm.RESOLVE_TREEWALK, vbm.RESOLVE_CACHED, vbm.RESOLVE_BRICK]
OUTPUTS = [vbm.OUTPUT_STREAMED, vbm.OUTPUT_MATERIALISED]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    gu.require_gpu()


@pytest.fixture(scope="module", params=sorted(SMALL))
def case(request):
    coords = SMALL[request.param]()
    return request.param, coords, oracle.OracleGrid(coords)


@pytest.mark.parametrize("method", ["select", "sweep"])
@pytest.mark.parametrize("log2w", [6, 7, 8, 9])
def test_decode(case, log2w, method):
    _, coords, o = case
    g = vbm.vbm_build(coords, log2w)
    li, vo = gu.decode(g, method)
    wli, wvo = o.decode(log2w)
    np.testing.assert_array_equal(li, wli)
    np.testing.assert_array_equal(vo, wvo)


@pytest.mark.parametrize("log2w", [7, 9])
@pytest.mark.parametrize("resolver", RESOLVERS)
def test_taps(case, log2w, resolver):
    _, coords, o = case
    g = vbm.vbm_build(coords, log2w)
    np.testing.assert_array_equal(gu.taps(g, 27, resolver), o.taps(27))
    np.testing.assert_array_equal(gu.taps(g, 7, resolver), o.taps(7))


@pytest.mark.parametrize("C", [1, 2, 3, 4, 5, 8, 13, 16])
def test_box_filter_all_variants(case, C):
    _, coords, o = case
    s = synth.sidecar_uniform(o.n, C, seed=C)
    want = gu.bits(o.box_filter(s, C))
    sd = gu.to_dev(s)
    for log2w in (6, 7, 9):
        g = vbm.vbm_build(coords, log2w)
        for r in RESOLVERS:
            for out in (OUTPUTS if r != vbm.RESOLVE_BRICK else OUTPUTS[:1]):
                got = gu.bits(gu.box_filter(g, sd, C, r, out))
                np.testing.assert_array_equal(got, want, err_msg=f"W=2^{log2w} resolver={r} output={out}")


@pytest.mark.parametrize("C", [32, 64])
@pytest.mark.parametrize("name", ["tiny_shell", "clusters"])
def test_wide_channels(name, C):
    # the widest sidecars (64 channels is the maximum C)
    coords = SMALL[name]()
    o = oracle.OracleGrid(coords)
    s = synth.sidecar_uniform(o.n, C, seed=C)
    sd = gu.to_dev(s)
    want = gu.bits(o.box_filter(s, C))
    want_lap = gu.bits(o.cross_filter(s, C, op=vbm.CROSS_LAPLACIAN))
    for log2w in (6, 9):
        g = vbm.vbm_build(coords, log2w)
        for r in RESOLVERS:
            np.testing.assert_array_equal(gu.bits(gu.box_filter(g, sd, C, r, vbm.OUTPUT_STREAMED)), want)
            np.testing.assert_array_equal(gu.bits(gu.cross_filter(g, sd, C, r, vbm.CROSS_LAPLACIAN)), want_lap)


@pytest.mark.parametrize("C", [1, 3, 8, 16])
@pytest.mark.parametrize("op", [vbm.CROSS_LAPLACIAN, vbm.CROSS_SUM])
def test_cross_filter(case, C, op):
    _, coords, o = case
    s = synth.sidecar_uniform(o.n, C, seed=100 + C)
    want = gu.bits(o.cross_filter(s, C, op=op))
    sd = gu.to_dev(s)
    for log2w in (6, 8):
        g = vbm.vbm_build(coords, log2w)
        for r in RESOLVERS:
            got = gu.bits(gu.cross_filter(g, sd, C, r, op))
            np.testing.assert_array_equal(got, want, err_msg=f"W=2^{log2w} resolver={r}")


def test_constant_sidecar_counts():
    coords = SMALL["tiny_shell"]()
    o = oracle.OracleGrid(coords)
    g = vbm.vbm_build(coords, 7)
    one = np.ones(o.n + 1, dtype=np.float32)
    one[0] = 0
    got = gu.box_filter(g, gu.to_dev(one), 1, vbm.RESOLVE_CACHED, vbm.OUTPUT_STREAMED)
    np.testing.assert_array_equal(got, o.box_filter(one, 1))
    assert got[0] == 0 and got[1:].min() >= 1 and got[1:].max() <= 27


def _phi(o, seed, background=0.75):
    rng = np.random.default_rng(seed)
    phi = rng.standard_normal(o.n + 1).astype(np.float32)
    phi[0] = background
    return phi


@pytest.mark.parametrize("log2w", [6, 7, 8, 9])
@pytest.mark.parametrize("resolver", RESOLVERS)
def test_weno(case, log2w, resolver):
    _, coords, o = case
    g = vbm.vbm_build(coords, log2w)
    np.testing.assert_array_equal(gu.taps(g, 19, resolver), o.taps(19))
    phi = _phi(o, seed=log2w)
    got = gu.weno_filter(g, gu.to_dev(phi), resolver, iso=0.1)
    np.testing.assert_array_equal(gu.bits(got), gu.bits(o.weno_filter(phi, iso=0.1)))


@pytest.mark.parametrize("resolver", RESOLVERS)
def test_weno_integer_field_and_ties(case, resolver):
    # integer-valued phi: some centres equal iso exactly (the inside branch)
    _, coords, o = case
    g = vbm.vbm_build(coords, 7)
    c = o.coords()
    phi = np.zeros(o.n + 1, dtype=np.float32)
    phi[1:] = (c[:, 0] + 2 * c[:, 1] - c[:, 2]) % 7 - 3
    phi[0] = 5.0
    want = o.weno_filter(phi, iso=0.0)
    np.testing.assert_array_equal(gu.bits(gu.weno_filter(g, gu.to_dev(phi), resolver, iso=0.0)), gu.bits(want))


@pytest.mark.parametrize("C", [8, 16, 24])
def test_box_16_byte_aligned_buffers(C):
    # sidecar and output 16- but not 32-byte aligned: the float4 lanes run
    # instead of the 256-bit ones, with the same bits
    t = gu.torch()
    coords = SMALL["tiny_shell"]()
    o = oracle.OracleGrid(coords)
    g = vbm.vbm_build(coords, 7)
    s = synth.sidecar_uniform(o.n, C, seed=2)
    want = gu.bits(o.box_filter(s, C))
    m = (o.n + 1) * C
    sbuf = t.zeros(m + 8, dtype=t.float32, device="cuda")
    obuf = t.full((m + 8,), float("nan"), dtype=t.float32, device="cuda")
    assert sbuf.data_ptr() % 32 == 0 and obuf.data_ptr() % 32 == 0
    for shift in (0, 4):
        sbuf[shift:shift + m] = t.from_numpy(s).cuda()
        vbm.vbm_box_filter(g, sbuf[shift:shift + m], C, obuf[shift:shift + m], vbm.RESOLVE_BRICK)
        t.cuda.synchronize()
        np.testing.assert_array_equal(gu.bits(obuf[shift:shift + m].cpu().numpy()), want)


@pytest.mark.parametrize("widths", [(1, 3, 8, 16), (16, 1), (5, 2, 13, 4), (8,), (3, 1), (2, 3, 8), (1, 2, 3),
                                    (16, 8), (3, 2, 1, 3, 2, 1, 16, 8)])
@pytest.mark.parametrize("resolver", RESOLVERS)
def test_box_filter_batch(case, widths, resolver):
    # one call filtering several sidecars equals the oracle's box filter of each,
    # bit for bit on every element; with the brick resolver the widths
    # 1/2/3/4/8/16 share a launch (up to four per launch), and two one-lane
    # widths (C <= 3) share one pass: the sets cover every such pair, in either
    # order, and a second launch
    t = gu.torch()
    _, coords, o = case
    hosts = [synth.sidecar_uniform(o.n, C, seed=10 + i) for i, C in enumerate(widths)]
    wants = [gu.bits(o.box_filter(h, C)) for h, C in zip(hosts, widths)]
    for log2w in (6, 9):
        g = vbm.vbm_build(coords, log2w)
        sides = [gu.to_dev(h) for h in hosts]
        outs = [t.full_like(s, float("nan")) for s in sides]
        vbm.vbm_box_filter_batch(g, sides, list(widths), outs, resolver)
        t.cuda.synchronize()
        for C, out, want in zip(widths, outs, wants):
            np.testing.assert_array_equal(gu.bits(out.cpu().numpy()), want, err_msg=f"C={C} W=2^{log2w}")


def test_box_filter_batch_errors():
    t = gu.torch()
    g = vbm.vbm_build(SMALL["tiny_shell"](), 7)
    s = t.zeros(g.n + 1, device="cuda")
    o = t.zeros(g.n + 1, device="cuda")
    with pytest.raises(vbm.VbmError):
        vbm.vbm_box_filter_batch(g, [], [], [])
    with pytest.raises(vbm.VbmError):
        vbm.vbm_box_filter_batch(g, [s] * 9, [1] * 9, [o] * 9)
    with pytest.raises(vbm.VbmError):  # two outputs alias
        vbm.vbm_box_filter_batch(g, [s, s], [1, 1], [o, o])
    s2 = t.zeros(g.n + 1, device="cuda")
    with pytest.raises(vbm.VbmError):  # an output is another entry's sidecar
        vbm.vbm_box_filter_batch(g, [s, s2], [1, 1], [s2, o])
    # partial overlaps: views of one buffer at different 16-byte offsets
    big = t.zeros(4 * (g.n + 1) + 64, device="cuda")
    a, b = big[: g.n + 1], big[4: g.n + 5]
    c3 = big[8: 8 + 3 * (g.n + 1)]
    with pytest.raises(vbm.VbmError, match="overlap"):  # two outputs share rows
        vbm.vbm_box_filter_batch(g, [s, s2], [1, 1], [a, b])
    with pytest.raises(vbm.VbmError, match="overlap"):  # an output shares rows with another entry's sidecar
        vbm.vbm_box_filter_batch(g, [s, a], [1, 1], [o, b])
    with pytest.raises(vbm.VbmError, match="overlap"):  # widths differ: C=3 output over a C=1 sidecar
        vbm.vbm_box_filter_batch(g, [a, t.zeros(3 * (g.n + 1), device="cuda")], [1, 3], [o, c3])
    # sidecars may share memory: both entries read the same rows
    o2 = t.zeros(g.n + 1, device="cuda")
    vbm.vbm_box_filter_batch(g, [a, a], [1, 1], [o, o2], vbm.RESOLVE_BRICK)
    t.cuda.synchronize()
    assert t.equal(o, o2)


def test_empty_grid():
    t = gu.torch()
    g = vbm.vbm_build(np.zeros((0, 3), dtype=np.int32), 7)
    assert g.n == 0 and g.n_slots == 0
    s = t.zeros(3, device="cuda")
    out = t.full((3,), 5.0, device="cuda")
    vbm.vbm_box_filter(g, s, 3, out)
    vbm.vbm_cross_filter(g, s, 3, out)
    taps = t.full((27,), 9, dtype=t.int32, device="cuda")
    vbm.vbm_box_taps(g, taps)
    lib = vbm.load()
    wout = t.full((1,), 5.0, device="cuda")
    vbm.vbm_weno_filter(g, s[:1], wout, 0.0, vbm.RESOLVE_BRICK)
    wtaps = t.full((19,), 9, dtype=t.int32, device="cuda")
    vbm.vbm_weno_taps(g, wtaps)
    t.cuda.synchronize()
    assert (wout.cpu() == 0).all() and (wtaps.cpu() == 0).all()
    assert lib.vbm_decode(g.handle, None, None, None) == 0  # no slots: nothing to write
    assert lib.vbm_decode_sweep(g.handle, None, None, None) == 0
    t.cuda.synchronize()
    assert (out.cpu() == 0).all() and (taps.cpu() == 0).all()


def test_device_errors():
    t = gu.torch()
    coords = SMALL["tiny_shell"]()
    g = vbm.vbm_build(coords, 7)
    n = g.n
    buf = t.zeros(n + 2, dtype=t.float32, device="cuda")
    lib = vbm.load()
    import ctypes
    buf2 = t.zeros(n + 2, dtype=t.float32, device="cuda")
    mis = ctypes.c_void_p(buf.data_ptr() + 4)
    ok = ctypes.c_void_p(buf.data_ptr())
    ok2 = ctypes.c_void_p(buf2.data_ptr())
    assert lib.vbm_box_filter(g.handle, mis, 1, ok, 1, 0, None) == -6
    assert lib.vbm_box_filter(g.handle, ok, 0, ok, 1, 0, None) == -1
    assert lib.vbm_box_filter(g.handle, ok, 65, ok, 1, 0, None) == -1
    assert lib.vbm_box_filter(g.handle, ok, 1, ok, 1, 0, None) == -1  # aliasing
    big = t.zeros(n + 1 + 8, dtype=t.float32, device="cuda")
    part = ctypes.c_void_p(big.data_ptr() + 16)  # aligned, shares all but 4 rows with big
    assert lib.vbm_box_filter(g.handle, ctypes.c_void_p(big.data_ptr()), 1, part, 1, 0, None) == -1
    assert b"overlaps" in lib.vbm_last_error()
    assert lib.vbm_weno_filter(g.handle, part, 0.0, ctypes.c_void_p(big.data_ptr()), 1, None) == -1
    assert lib.vbm_box_filter(g.handle, ok, 1, mis, 7, 0, None) == -1
    assert lib.vbm_cross_filter(g.handle, ok, 1, ok2, 1, 5, None) == -1
    assert b"op" in lib.vbm_last_error()
    assert lib.vbm_weno_filter(g.handle, mis, 0.0, ok2, 1, None) == -6
    assert lib.vbm_weno_filter(g.handle, ok, 0.0, ok, 1, None) == -1  # aliasing
    assert lib.vbm_weno_filter(g.handle, ok, 0.0, ok2, 9, None) == -1
    assert lib.vbm_weno_taps(g.handle, ok, 9, None) == -1
    assert lib.vbm_weno_taps(g.handle, None, 0, None) == -1
    for fn in (lib.vbm_decode, lib.vbm_decode_sweep):
        assert fn(g.handle, None, ok, None) == -1
        assert fn(g.handle, mis, ok, None) == -6
        assert fn(g.handle, ok, mis, None) == -6


@pytest.mark.parametrize("resolver", [vbm.RESOLVE_BRICK, vbm.RESOLVE_CACHED])
def test_box_filter_batch_host_matches_oracle(resolver):
    """vbm_box_filter_batch_host (host sidecars in, host outputs back) equals
    the oracle on every element, on three calls in a row with new data each
    time (the grid's two staging sets used, then reused), with pinned torch
    tensors and with pageable numpy arrays; a wider batch grows the staging."""
    t = gu.torch()
    coords = SMALL["tiny_shell"]()
    o = oracle.OracleGrid(coords)
    g = vbm.vbm_build(coords, 7)
    widths = (1, 3, 8, 16)
    for call in range(3):
        pinned = call != 1
        hosts = [synth.sidecar_uniform(o.n, C, seed=100 * call + C) for C in widths]
        if pinned:
            ins = [t.from_numpy(h).pin_memory() for h in hosts]
            outs = [t.full((len(h),), float("nan")).pin_memory() for h in hosts]
        else:
            ins = hosts
            outs = [np.full(len(h), np.nan, dtype=np.float32) for h in hosts]
        vbm.vbm_box_filter_batch_host(g, ins, list(widths), outs, resolver)
        t.cuda.current_stream().synchronize()
        for h, C, out in zip(hosts, widths, outs):
            got = out.numpy() if pinned else out
            np.testing.assert_array_equal(gu.bits(got), gu.bits(o.box_filter(h, C)), err_msg=f"call {call} C={C}")
    wide = (5, 24, 64)  # widths outside the fused layouts, and a larger staging set
    hosts = [synth.sidecar_uniform(o.n, C, seed=7 + C) for C in wide]
    outs = [np.empty_like(h) for h in hosts]
    vbm.vbm_box_filter_batch_host(g, hosts, list(wide), outs, resolver)
    t.cuda.current_stream().synchronize()
    for h, C, out in zip(hosts, wide, outs):
        np.testing.assert_array_equal(gu.bits(out), gu.bits(o.box_filter(h, C)), err_msg=f"C={C}")
    g.close()


def test_box_filter_batch_host_back_to_back():
    """Five host-buffer calls enqueued back to back with no synchronisation
    between them, each with its own pinned inputs and outputs: calls i and
    i+2 reuse one staging set, so every output is correct only if each reuse
    waits for the set's previous filter and copies back."""
    t = gu.torch()
    coords = SMALL["tiny_shell"]()
    o = oracle.OracleGrid(coords)
    g = vbm.vbm_build(coords, 9)
    widths = (1, 3, 8, 16)
    calls = []
    for call in range(5):
        hosts = [synth.sidecar_uniform(o.n, C, seed=1000 * call + C) for C in widths]
        ins = [t.from_numpy(h).pin_memory() for h in hosts]
        outs = [t.full((len(h),), float("nan")).pin_memory() for h in hosts]
        vbm.vbm_box_filter_batch_host(g, ins, list(widths), outs, vbm.RESOLVE_BRICK)
        calls.append((hosts, outs))
    t.cuda.current_stream().synchronize()
    for call, (hosts, outs) in enumerate(calls):
        for h, C, out in zip(hosts, widths, outs):
            np.testing.assert_array_equal(gu.bits(out.numpy()), gu.bits(o.box_filter(h, C)),
                                          err_msg=f"call {call} C={C}")
    g.close()


def test_box_filter_batch_host_errors_and_empty_grid():
    t = gu.torch()
    g = vbm.vbm_build(SMALL["tiny_shell"](), 7)
    h = np.zeros(g.n + 1, dtype=np.float32)
    with pytest.raises(vbm.VbmError, match="overlap"):  # an output over the sidecar
        vbm.vbm_box_filter_batch_host(g, [h], [1], [h])
    big = np.zeros(2 * (g.n + 1), dtype=np.float32)
    with pytest.raises(vbm.VbmError, match="overlap"):  # two outputs share rows
        vbm.vbm_box_filter_batch_host(g, [h, h], [1, 1], [big[: g.n + 1], big[3: g.n + 4]])
    lib = vbm.load()
    import ctypes
    arr = (ctypes.c_void_p * 1)(None)
    cs = (ctypes.c_int * 1)(1)
    assert lib.vbm_box_filter_batch_host(g.handle, 1, arr, cs, arr, vbm.RESOLVE_BRICK, None) == -1
    assert b"NULL" in lib.vbm_last_error()
    assert lib.vbm_box_filter_batch_host(g.handle, 0, arr, cs, arr, vbm.RESOLVE_BRICK, None) == -1
    e = vbm.vbm_build(np.zeros((0, 3), dtype=np.int32), 7)
    ins = [np.ones(3, dtype=np.float32)]
    outs = [np.full(3, 5.0, dtype=np.float32)]
    vbm.vbm_box_filter_batch_host(e, ins, [3], outs)
    t.cuda.current_stream().synchronize()
    assert (outs[0] == 0).all()


def test_probe_launch():
    """The measurement probes run with the filters' launch shape and leave the
    grid and the sidecar untouched; bad arguments are rejected."""
    t = gu.torch()
    g = vbm.vbm_build(SMALL["tiny_shell"](), 7)
    s = gu.to_dev(synth.sidecar_uniform(g.n, 1, seed=3))
    before = s.clone()
    for kind in (vbm.PROBE_EMPTY, vbm.PROBE_METADATA, vbm.PROBE_CHAIN):
        vbm.vbm_probe_launch(g, kind, s)
    t.cuda.synchronize()
    assert t.equal(s, before)
    lib = vbm.load()
    assert lib.vbm_probe_launch(g.handle, 3, None, None) == -1
    assert lib.vbm_probe_launch(g.handle, vbm.PROBE_CHAIN, None, None) == -1
    assert lib.vbm_probe_launch(None, vbm.PROBE_EMPTY, None, None) == -1
