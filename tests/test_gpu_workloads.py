"""GPU parity at full workload sizes.

Shell S185 (183.5 <= |p| <= 186.5, 1,290,538 voxels), the decode grid D
(random 8^3 bricks on 512^3, ~20.4M voxels) and the fog F (value noise on
512^3, ~42.9M voxels).  Decode maps are compared with the oracle in full.  The
benchmarked call (the device-built shell, W=512, four sidecars in one batched
call) is compared with the oracle on every element, the oracle running on all
host cores; other filter outputs on sampled voxels (every voxel of the fog's
blocks that span more than MaxCachedLeaves leaves included), and all
resolver/output variants must agree bit for bit on every voxel.
"""
import numpy as np
import pytest

import oracle
import sparse_voxel_grid_gb300 as vbm
import synth
from tests import gpu_util as gu
from tests import oracle_pool

pytestmark = pytest.mark.gpu

RESOLVERS = [vbm.RESOLVE_TREEWALK, vbm.RESOLVE_CACHED, vbm.RESOLVE_BRICK]
OUTPUTS = [vbm.OUTPUT_STREAMED, vbm.OUTPUT_MATERIALISED]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    gu.require_gpu()


def _sample(n, k=20000, seed=0):
    rng = np.random.default_rng(seed)
    idx = np.concatenate([np.arange(1, min(n, 600) + 1), np.arange(max(1, n - 600), n + 1),
                          rng.integers(1, n + 1, size=k)])
    return np.unique(idx)


@pytest.fixture(scope="module")
def shell():
    coords = synth.WORKLOADS["S185"]()
    return coords, oracle.OracleGrid(coords)


@pytest.mark.parametrize("method", ["select", "sweep"])
@pytest.mark.parametrize("log2w", [6, 7, 8, 9])
def test_shell_decode_full(shell, log2w, method):
    coords, o = shell
    g = vbm.vbm_build(coords, log2w)
    li, vo = gu.decode(g, method)
    wli, wvo = o.decode(log2w)
    np.testing.assert_array_equal(li, wli)
    np.testing.assert_array_equal(vo, wvo)


@pytest.mark.parametrize("log2w", [7, 9])
def test_shell_taps(shell, log2w):
    coords, o = shell
    g = vbm.vbm_build(coords, log2w)
    which = _sample(o.n)
    for shape in (27, 7):
        walk = gu.taps(g, shape, vbm.RESOLVE_TREEWALK)
        cached = gu.taps(g, shape, vbm.RESOLVE_CACHED)
        np.testing.assert_array_equal(walk, cached)
        np.testing.assert_array_equal(gu.taps(g, shape, vbm.RESOLVE_BRICK), cached)
        np.testing.assert_array_equal(cached[which], o.taps(shape, which=which))
        assert (cached[0] == 0).all()


@pytest.mark.parametrize("C", [1, 3, 8, 16])
@pytest.mark.parametrize("log2w", [7, 9])
def test_shell_box_filter(shell, C, log2w):
    coords, o = shell
    g = vbm.vbm_build(coords, log2w)
    s = synth.sidecar_uniform(o.n, C, seed=0)
    sd = gu.to_dev(s)
    ref = gu.bits(gu.box_filter(g, sd, C, vbm.RESOLVE_CACHED, vbm.OUTPUT_STREAMED))
    for r in RESOLVERS:
        for out in (OUTPUTS if r != vbm.RESOLVE_BRICK else OUTPUTS[:1]):
            if (r, out) == (vbm.RESOLVE_CACHED, vbm.OUTPUT_STREAMED):
                continue
            np.testing.assert_array_equal(gu.bits(gu.box_filter(g, sd, C, r, out)), ref)
    which = _sample(o.n, k=4000 if C > 3 else 20000, seed=C)
    want = gu.bits(o.box_filter(s, C, which=which)).reshape(-1, C)
    np.testing.assert_array_equal(ref.reshape(-1, C)[which], want)
    assert (ref[:C] == 0).all()


def test_shell_box_filter_batch(shell):
    # the benchmarked call: four sidecars in one launch, bit for bit as four calls
    coords, o = shell
    t = gu.torch()
    g = vbm.vbm_build(coords, 9)
    sides = [gu.to_dev(synth.sidecar_uniform(o.n, C, seed=0)) for C in (1, 3, 8, 16)]
    outs = [t.full_like(s, float("nan")) for s in sides]
    vbm.vbm_box_filter_batch(g, sides, [1, 3, 8, 16], outs, vbm.RESOLVE_BRICK)
    t.cuda.synchronize()
    for s, C, out in zip(sides, (1, 3, 8, 16), outs):
        want = gu.bits(gu.box_filter(g, s, C, vbm.RESOLVE_BRICK, vbm.OUTPUT_STREAMED))
        np.testing.assert_array_equal(gu.bits(out.cpu().numpy()), want, err_msg=f"C={C}")


def test_shell_benchmarked_call_every_element(shell):
    """The benchmarked configuration exactly: the grid built on the device at
    W=512, sidecars U[-1,1) seed 0 at C = 1, 3, 8, 16 in one
    vbm_box_filter_batch call (brick resolver), every output element against
    the oracle."""
    coords, o = shell
    t = gu.torch()
    cs = (1, 3, 8, 16)
    g = vbm.vbm_build_device(t.from_numpy(coords).cuda(), 9)
    assert g.n == o.n
    sides = [gu.to_dev(synth.sidecar_uniform(o.n, C, seed=0)) for C in cs]
    outs = [t.full_like(s, float("nan")) for s in sides]
    vbm.vbm_box_filter_batch(g, sides, list(cs), outs, vbm.RESOLVE_BRICK)
    t.cuda.synchronize()
    wants = oracle_pool.box_filter_all("S185", o.n, cs, seeds=(0, 0, 0, 0))
    for C, out, want in zip(cs, outs, wants):
        np.testing.assert_array_equal(gu.bits(out.cpu().numpy()), gu.bits(want), err_msg=f"C={C}")


def test_shell_laplacian(shell):
    coords, o = shell
    s = synth.sidecar_uniform(o.n, 1, seed=0)
    want = gu.bits(o.cross_filter(s, 1, op=vbm.CROSS_LAPLACIAN))
    sd = gu.to_dev(s)
    for log2w in (6, 7, 8, 9):
        g = vbm.vbm_build(coords, log2w)
        for r in RESOLVERS:
            got = gu.bits(gu.cross_filter(g, sd, 1, r, vbm.CROSS_LAPLACIAN))
            np.testing.assert_array_equal(got, want, err_msg=f"W=2^{log2w} resolver={r}")


def _level_set(o, background=3.0):
    """phi = |p| - 185 (the shell's signed distance), row 0 the background."""
    c = o.coords().astype(np.float64)
    phi = np.empty(o.n + 1, dtype=np.float32)
    phi[1:] = (np.sqrt((c ** 2).sum(1)) - 185.0).astype(np.float32)
    phi[0] = background
    return phi


def test_shell_weno(shell):
    coords, o = shell
    phi = _level_set(o)
    want = gu.bits(o.weno_filter(phi, iso=0.0))
    pd = gu.to_dev(phi)
    for log2w in (6, 7, 8, 9):
        g = vbm.vbm_build(coords, log2w)
        for r in RESOLVERS:
            got = gu.bits(gu.weno_filter(g, pd, r, iso=0.0))
            np.testing.assert_array_equal(got, want, err_msg=f"W=2^{log2w} resolver={r}")
        if log2w in (7, 9):
            taps = gu.taps(g, 19, vbm.RESOLVE_BRICK)
            np.testing.assert_array_equal(taps, gu.taps(g, 19, vbm.RESOLVE_CACHED))
            which = _sample(o.n, k=5000, seed=log2w)
            np.testing.assert_array_equal(taps[which], o.taps(19, which=which))


@pytest.fixture(scope="module")
def bricks():
    coords = synth.WORKLOADS["D"]()
    return coords, oracle.OracleGrid(coords)


@pytest.mark.parametrize("method", ["select", "sweep"])
@pytest.mark.parametrize("log2w", [6, 7, 8, 9])
def test_decode_grid_full(bricks, log2w, method):
    coords, o = bricks
    g = vbm.vbm_build(coords, log2w)
    li, vo = gu.decode(g, method)
    wli, wvo = o.decode(log2w)
    np.testing.assert_array_equal(li, wli)
    np.testing.assert_array_equal(vo, wvo)
    sent = li == vbm.SENTINEL_LEAF
    assert sent.sum() == g.n_slots - o.n


def test_decode_grid_box_filter_batch(bricks):
    # the benchmarked call on the dense-leaf grid D (20.4M voxels, W=512): every
    # output against the width filtered alone by the cached resolver, and a
    # sample of each against the oracle
    coords, o = bricks
    t = gu.torch()
    g = vbm.vbm_build(coords, 9)
    cs = (1, 3, 8, 16)
    host = {C: synth.sidecar_uniform(o.n, C, seed=40 + C) for C in cs}
    sides = [gu.to_dev(host[C]) for C in cs]
    outs = [t.full_like(s, float("nan")) for s in sides]
    vbm.vbm_box_filter_batch(g, sides, list(cs), outs, vbm.RESOLVE_BRICK)
    t.cuda.synchronize()
    which = _sample(o.n, k=3000, seed=4)
    for s, C, out in zip(sides, cs, outs):
        got = gu.bits(out.cpu().numpy())
        np.testing.assert_array_equal(got, gu.bits(gu.box_filter(g, s, C, vbm.RESOLVE_CACHED, vbm.OUTPUT_STREAMED)),
                                      err_msg=f"C={C}")
        want = gu.bits(o.box_filter(host[C], C, which=which)).reshape(-1, C)
        np.testing.assert_array_equal(got.reshape(-1, C)[which], want, err_msg=f"C={C} against the oracle")


def _over_cache_voxels(g, log2w):
    """Indices of every voxel of the blocks that span more than MaxCachedLeaves
    leaves (the cached resolver's tree-walk fallback)."""
    jm = vbm.vbm_leaf_export(g, "block_jump")
    spans = 1 + np.array([sum(bin(int(w)).count("1") for w in row) for row in jm])
    W = 1 << log2w
    blocks = np.nonzero(spans > vbm.MAX_CACHED_LEAVES)[0]
    idx = np.concatenate([np.arange(1 + b * W, 1 + (b + 1) * W) for b in blocks]) if len(blocks) else np.zeros(0)
    return blocks, idx[idx <= g.n].astype(np.int64)


@pytest.fixture(scope="module")
def fog():
    coords = synth.WORKLOADS["F"]()
    return coords, oracle.OracleGrid(coords)


def test_fog_box_filter(fog):
    coords, o = fog
    g = vbm.vbm_build(coords, 8)
    info = g.info
    assert info["n_active"] == o.n
    blocks, over = _over_cache_voxels(g, 8)
    assert len(blocks) == info["n_blocks_over_cache"] > 0
    C = 8
    s = synth.sidecar_normal(o.n, C, seed=0)
    sd = gu.to_dev(s)
    cached = gu.bits(gu.box_filter(g, sd, C, vbm.RESOLVE_CACHED, vbm.OUTPUT_STREAMED))
    walk = gu.bits(gu.box_filter(g, sd, C, vbm.RESOLVE_TREEWALK, vbm.OUTPUT_STREAMED))
    np.testing.assert_array_equal(cached, walk)
    brick = gu.bits(gu.box_filter(g, sd, C, vbm.RESOLVE_BRICK, vbm.OUTPUT_STREAMED))
    np.testing.assert_array_equal(brick, walk)
    # every voxel of the over-cache blocks, and a sample of 60k others
    which = np.union1d(_sample(o.n, k=60000), over)
    want = gu.bits(o.box_filter(s, C, which=which)).reshape(-1, C)
    np.testing.assert_array_equal(cached.reshape(-1, C)[which], want)


def test_fog_box_filter_batch(fog):
    coords, o = fog
    t = gu.torch()
    g = vbm.vbm_build_device(t.from_numpy(coords).cuda(), 8)
    _, over = _over_cache_voxels(g, 8)
    assert len(over) > 0
    hosts = {C: synth.sidecar_normal(g.n, C, seed=C) for C in (1, 8)}
    sides = [gu.to_dev(hosts[C]) for C in (1, 8)]
    outs = [t.full_like(s, float("nan")) for s in sides]
    vbm.vbm_box_filter_batch(g, sides, [1, 8], outs, vbm.RESOLVE_BRICK)
    t.cuda.synchronize()
    which = np.union1d(_sample(o.n, k=30000, seed=5), over)
    for s, C, out in zip(sides, (1, 8), outs):
        got = gu.bits(out.cpu().numpy())
        want = gu.bits(gu.box_filter(g, s, C, vbm.RESOLVE_CACHED, vbm.OUTPUT_STREAMED))
        np.testing.assert_array_equal(got, want, err_msg=f"C={C}")
        np.testing.assert_array_equal(got.reshape(-1, C)[which],
                                      gu.bits(o.box_filter(hosts[C], C, which=which)).reshape(-1, C),
                                      err_msg=f"C={C} against the oracle")


def test_fog_weno(fog):
    coords, o = fog
    g = vbm.vbm_build(coords, 8)
    phi = synth.sidecar_normal(o.n, 1, seed=3)
    phi[0] = 0.5
    pd = gu.to_dev(phi)
    cached = gu.bits(gu.weno_filter(g, pd, vbm.RESOLVE_CACHED))
    np.testing.assert_array_equal(gu.bits(gu.weno_filter(g, pd, vbm.RESOLVE_BRICK)), cached)
    np.testing.assert_array_equal(gu.bits(gu.weno_filter(g, pd, vbm.RESOLVE_TREEWALK)), cached)
    which = _sample(o.n, k=6000, seed=3)
    np.testing.assert_array_equal(cached[which], gu.bits(o.weno_filter(phi, which=which)))
