"""Host-side checks of the product's grid builder against the oracle (no GPU).

vbm_build with VBM_BUILD_HOST_ONLY makes no CUDA call; vbm_leaf_export copies
its arrays out.  These are compared with the oracle's enumeration of leaves,
decode and block metadata.
"""
import numpy as np
import pytest

import oracle
import sparse_voxel_grid_gb300 as vbm
import synth
from tests.test_oracle_pins import GRIDS


def _host_grid(coords, log2w, flags=0):
    return vbm.vbm_build(coords, log2w, flags | vbm.BUILD_HOST_ONLY)


CASES = ["tiny_shell", "clusters", "random_box", "cube"]


@pytest.fixture(scope="module", params=CASES)
def case(request):
    coords = GRIDS[request.param]()
    return coords, oracle.OracleGrid(coords)


def test_leaves_match_oracle(case):
    coords, o = case
    g = _host_grid(coords, 7)
    leaf_of, origins = o.leaves()
    info = g.info
    assert info["n_active"] == o.n
    assert info["n_leaves"] == len(origins)
    np.testing.assert_array_equal(vbm.vbm_leaf_export(g, "leaf_origin"), origins)
    first = vbm.vbm_leaf_export(g, "leaf_first").astype(np.int64)
    want_first = np.searchsorted(leaf_of[1:], np.arange(len(origins))) + 1
    np.testing.assert_array_equal(first, want_first)
    # masks: bit off%64 of word off//64 set exactly for the leaf's voxels
    masks = vbm.vbm_leaf_export(g, "leaf_mask")
    li, vo = o.decode(7)
    want = np.zeros((len(origins), 8), dtype=np.uint64)
    for L, off in zip(li[:o.n].tolist(), vo[:o.n].tolist()):
        want[L, off // 64] |= np.uint64(1) << np.uint64(off % 64)
    np.testing.assert_array_equal(masks, want)
    # 9-bit directory: field w-1 = set bits in words 0..w-1
    prefix = vbm.vbm_leaf_export(g, "leaf_prefix")
    counts = np.array([[bin(int(w)).count("1") for w in row] for row in masks])
    for w in range(1, 8):
        field = (prefix >> np.uint64(9 * (w - 1))) & np.uint64(511)
        np.testing.assert_array_equal(field.astype(np.int64), counts[:, :w].sum(axis=1))


def test_neighbour_rows(case):
    """Entry (dx+1)*9+(dy+1)*3+(dz+1) of leaf L is the leaf 8*(dx,dy,dz) away."""
    coords, o = case
    g = _host_grid(coords, 7)
    _, origins = o.leaves()
    where = {tuple(p): i for i, p in enumerate(origins.tolist())}
    nbr = vbm.vbm_leaf_export(g, "leaf_neighbours")
    assert nbr.shape == (len(origins), 32)
    assert (nbr[:, 27:] == 0xFFFFFFFF).all()
    for L, (x, y, z) in enumerate(origins.tolist()):
        for t in range(27):
            want = where.get((x + 8 * (t // 9 - 1), y + 8 * ((t // 3) % 3 - 1), z + 8 * (t % 3 - 1)), 0xFFFFFFFF)
            assert nbr[L, t] == want
        assert nbr[L, 13] == L


@pytest.mark.parametrize("log2w", [6, 7, 8, 9])
def test_block_metadata_matches_oracle(case, log2w):
    coords, o = case
    g = _host_grid(coords, log2w)
    fl, jm = o.blocks(log2w)
    np.testing.assert_array_equal(vbm.vbm_leaf_export(g, "block_first_leaf"), fl)
    np.testing.assert_array_equal(vbm.vbm_leaf_export(g, "block_jump"), jm)
    spans = 1 + np.array([sum(bin(int(w)).count("1") for w in row) for row in jm], dtype=np.int64)
    info = g.info
    assert info["max_span"] == (spans.max() if len(spans) else 0)
    assert info["n_blocks_over_cache"] == int((spans > vbm.MAX_CACHED_LEAVES).sum())


def test_dedup_and_duplicates():
    c = np.array([[0, 0, 0], [1, 2, 3], [0, 0, 0], [9, 9, 9]], dtype=np.int32)
    with pytest.raises(vbm.VbmError) as e:
        _host_grid(c, 7)
    assert e.value.code == -2
    g = _host_grid(c, 7, vbm.BUILD_DEDUP)
    assert g.n == 3
    o = oracle.OracleGrid(np.unique(c, axis=0))
    np.testing.assert_array_equal(vbm.vbm_leaf_export(g, "leaf_origin"), o.leaves()[1])


def test_empty_grid():
    g = _host_grid(np.zeros((0, 3), dtype=np.int32), 7)
    info = g.info
    assert info["n_active"] == 0 and info["n_blocks"] == 0 and info["n_leaves"] == 0


def test_coordinate_range():
    with pytest.raises(vbm.VbmError) as e:
        _host_grid(np.array([[2 ** 30 + 1, 0, 0]], dtype=np.int32), 7)
    assert e.value.code == -3
    g = _host_grid(np.array([[2 ** 30, -2 ** 30, 5]], dtype=np.int32), 7)
    assert g.n == 1


def test_fallback_grid_spans_many_leaves():
    """One voxel per leaf: every full block spans W leaves (> MaxCachedLeaves)."""
    c = synth.scatter(side=12, count=1000, origin=-40, seed=3)
    g = _host_grid(c, 7)
    info = g.info
    assert info["n_leaves"] == 1000
    assert info["max_span"] == 128
    assert info["n_blocks_over_cache"] == 8  # 7 full blocks and a last block of 104 leaves


@pytest.mark.slow
def test_workload_shapes():
    """The shell workloads: counts the builder reports (S160 reproduces the
    pages' 9140 leaves)."""
    g = _host_grid(synth.WORKLOADS["S160"](), 7)
    assert g.info["n_leaves"] == 9140 and g.info["n_active"] == 1288594
    g = _host_grid(synth.WORKLOADS["S185"](), 7)
    assert g.info["n_active"] == 1290538 and g.info["n_leaves"] == 11255
    assert g.info["n_blocks_over_cache"] == 0
