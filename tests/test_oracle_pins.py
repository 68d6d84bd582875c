"""Pins of the CPU oracle against things other than itself (no GPU needed).

Each check uses a formulation the oracle does not: a nested-dictionary tree
walk and dictionary stencil lookups (tests/bruteforce.py), closed forms on
full cubes, pair counting, and the counts the pages print for their workload.
The readings of the pages that these pin are listed in oracle/oracle.cpp.
"""
import os

import numpy as np
import pytest

import oracle
import synth
from tests import bruteforce as bf

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    vals = {}
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        parts = line.split()
        vals[parts[0]] = [float(v) for v in parts[1:]]
    return vals


def _clusters(seed=1):
    """Small random clusters straddling upper-node (4096) and lower-node (128)
    boundaries, on both sides of zero, plus a few far-away points."""
    centres = [(-4096, 0, 4095), (127, -129, 0), (0, 0, 0), (4095, 4096, -1), (-1, -8, 7)]
    parts = [synth.dense_random((6, 7, 5), 0.45, seed=seed + i, origin=(cx - 3, cy - 3, cz - 2))
             for i, (cx, cy, cz) in enumerate(centres)]
    parts.append(np.array([[1_000_000, -2_000_000, 5], [-70_000, 33, 9_999], [8, 8, 8]], dtype=np.int32))
    pts = np.concatenate(parts)
    return np.unique(pts, axis=0).astype(np.int32)


def _cube(side=10, origin=(-5, -5, -5)):
    r = np.arange(side)
    g = np.stack(np.meshgrid(r, r, r, indexing="ij"), axis=-1).reshape(-1, 3)
    return (g + np.asarray(origin)).astype(np.int32)


GRIDS = {
    "tiny_shell": lambda: synth.WORKLOADS["T"](),
    "clusters": _clusters,
    "random_box": lambda: synth.dense_random((14, 13, 15), 0.3, seed=7, origin=(-7, 3, -2)),
    "cube": _cube,
}


@pytest.fixture(scope="module", params=sorted(GRIDS))
def grid(request):
    coords = GRIDS[request.param]()
    g = oracle.OracleGrid(coords)
    d = bf.Dense(bf.tree_order(coords))
    return request.param, coords, g, d


def _bits(a):
    return np.asarray(a, dtype=np.float32).view(np.uint32)


# ---------------------------------------------------------------------------
# Index assignment (tree order)
# ---------------------------------------------------------------------------

def test_tree_order_matches_nested_walk(grid):
    _, coords, g, d = grid
    assert g.n == len(coords)
    np.testing.assert_array_equal(g.coords().astype(np.int64), d.ordered)


def test_index_lookup_is_inverse(grid):
    _, coords, g, d = grid
    rng = np.random.default_rng(0)
    for i in rng.choice(np.arange(1, g.n + 1), size=min(200, g.n), replace=False):
        x, y, z = d.ordered[i - 1]
        assert g.index(int(x), int(y), int(z)) == i
    # points that are not active
    lo = d.lo
    for _ in range(200):
        p = lo + rng.integers(0, np.asarray(d.shape))
        want = d.lookup(p[None, :])[0]
        assert g.index(int(p[0]), int(p[1]), int(p[2])) == want


def test_duplicates_rejected():
    c = np.array([[0, 0, 0], [1, 2, 3], [0, 0, 0]], dtype=np.int32)
    with pytest.raises(ValueError):
        oracle.OracleGrid(c)


# ---------------------------------------------------------------------------
# Stencil taps and filters against the dense volume
# ---------------------------------------------------------------------------

def test_box_taps_match_dense(grid):
    _, _, g, d = grid
    t = g.taps(27)
    assert (t[0] == 0).all()
    np.testing.assert_array_equal(t[1:].astype(np.int64), d.box_taps())
    assert (t[1:, 13] == np.arange(1, g.n + 1)).all()  # the centre tap is the voxel itself


def test_cross_taps_match_dense(grid):
    _, _, g, d = grid
    t = g.taps(7)
    np.testing.assert_array_equal(t[1:].astype(np.int64), d.cross_taps())
    # the cross is the box restricted to taps 4,10,12,13,14,16,22
    np.testing.assert_array_equal(t, g.taps(27)[:, list(oracle.CROSS_TAPS)])


@pytest.mark.parametrize("C", [1, 3, 8])
def test_box_filter_bitexact_dense(grid, C):
    _, _, g, d = grid
    s = synth.sidecar_uniform(g.n, C, seed=11)
    out = g.box_filter(s, C).reshape(-1, C)
    assert (_bits(out[0]) == 0).all()
    np.testing.assert_array_equal(_bits(out[1:]), _bits(d.box_filter(s, C)))


@pytest.mark.parametrize("C", [1, 3])
def test_laplacian_bitexact_dense(grid, C):
    _, _, g, d = grid
    s = synth.sidecar_uniform(g.n, C, seed=5)
    out = g.cross_filter(s, C, op=0).reshape(-1, C)
    np.testing.assert_array_equal(_bits(out[1:]), _bits(d.laplacian(s, C)))


def test_cross_sum_bitexact_dense(grid):
    _, _, g, d = grid
    s = synth.sidecar_uniform(g.n, 2, seed=3)
    out = g.cross_filter(s, 2, op=1).reshape(-1, 2)
    rows = s.reshape(-1, 2)
    acc = np.zeros((g.n, 2), dtype=np.float32)
    for j in range(7):
        nb = d.cross_taps()[:, j]
        v = rows[nb].copy()
        v[nb == 0] = 0.0
        acc = acc + v
    np.testing.assert_array_equal(_bits(out[1:]), _bits(acc))


def test_tap_order_matters_and_is_pinned():
    """The pin above is sensitive to summation order: summing the same taps in
    reverse order changes some fp32 results on a random sidecar."""
    coords = GRIDS["random_box"]()
    d = bf.Dense(bf.tree_order(coords))
    s = synth.sidecar_uniform(d.n, 1, seed=11)
    fwd = d.box_filter(s, 1)
    rows = s.reshape(-1, 1)
    rev = np.zeros_like(fwd)
    for di in (1, 0, -1):
        for dj in (1, 0, -1):
            for dk in (1, 0, -1):
                nb = d.neighbour(di, dj, dk)
                v = rows[nb].copy()
                v[nb == 0] = 0.0
                rev = rev + v
    assert (_bits(fwd) != _bits(rev)).any()


def test_integer_sidecar_pins_resolution(grid):
    """With integer values (exact in fp32) the sum is order-free: this checks
    which neighbours are found separately from the summation order."""
    _, _, g, d = grid
    xyz = g.coords().astype(np.int64)
    f = np.mod(7 * xyz[:, 0] + 13 * xyz[:, 1] + 29 * xyz[:, 2], 1021)  # small: sums exact in fp32
    s = np.concatenate([[0.0], f]).astype(np.float32)
    out = g.box_filter(s, 1)[1:].astype(np.float64)
    occ_sum = np.zeros(g.n, dtype=np.float64)
    for di in (-1, 0, 1):
        for dj in (-1, 0, 1):
            for dk in (-1, 0, 1):
                nb = d.neighbour(di, dj, dk)
                occ_sum += np.where(nb > 0, s.astype(np.float64)[nb], 0.0)
    np.testing.assert_array_equal(out, occ_sum)


# ---------------------------------------------------------------------------
# Closed forms and invariants
# ---------------------------------------------------------------------------

def _neighbour_counts(d):
    cnt = np.zeros(d.n, dtype=np.int64)
    for di in (-1, 0, 1):
        for dj in (-1, 0, 1):
            for dk in (-1, 0, 1):
                cnt += d.neighbour(di, dj, dk) > 0
    return cnt


def test_constant_one_counts_neighbours(grid):
    _, _, g, d = grid
    one = np.ones(g.n + 1, dtype=np.float32)
    one[0] = 0.0
    box = g.box_filter(one, 1)[1:]
    np.testing.assert_array_equal(box.astype(np.int64), _neighbour_counts(d))
    lap = g.cross_filter(one, 1, op=0)[1:]
    faces = sum((d.neighbour(a, b, c) > 0).astype(np.int64) for a, b, c in bf.Dense.FACES)
    np.testing.assert_array_equal(lap.astype(np.int64), faces.astype(np.int64) - 6)


def test_full_cube_closed_forms():
    n = 10
    g = oracle.OracleGrid(_cube(n, (-5, -5, -5)))
    one = np.ones(g.n + 1, dtype=np.float32)
    one[0] = 0.0
    box = g.box_filter(one, 1)[1:]
    vals, counts = np.unique(box, return_counts=True)
    assert dict(zip(vals.tolist(), counts.tolist())) == {8.0: 8, 12.0: 12 * (n - 2), 18.0: 6 * (n - 2) ** 2,
                                                         27.0: (n - 2) ** 3}
    lap = g.cross_filter(one, 1, op=0)[1:]
    vals, counts = np.unique(lap, return_counts=True)
    assert dict(zip(vals.tolist(), counts.tolist())) == {-3.0: 8, -2.0: 12 * (n - 2), -1.0: 6 * (n - 2) ** 2,
                                                         0.0: (n - 2) ** 3}
    # a linear field: interior box sums are 27 * f(centre); interior Laplacian is 0
    xyz = g.coords().astype(np.int64)
    f = (xyz[:, 0] + 2 * xyz[:, 1] + 3 * xyz[:, 2]) + 100
    s = np.concatenate([[0.0], f]).astype(np.float32)
    interior = np.all((xyz > -5) & (xyz < 4), axis=1)
    box = g.box_filter(s, 1)[1:]
    np.testing.assert_array_equal(box[interior], 27.0 * f[interior])
    lap = g.cross_filter(s, 1, op=0)[1:]
    assert (lap[interior] == 0.0).all()


def test_pair_symmetry():
    """Sum over voxels of the box of 1 = N + 2P, P = unordered pairs of distinct
    voxels at Chebyshev distance 1 (counted over all pairs)."""
    coords = synth.dense_random((9, 8, 9), 0.35, seed=21, origin=(-4, -4, 3))
    g = oracle.OracleGrid(coords)
    one = np.ones(g.n + 1, dtype=np.float32)
    one[0] = 0.0
    total = g.box_filter(one, 1)[1:].astype(np.int64).sum()
    c = coords.astype(np.int64)
    cheb = np.abs(c[:, None, :] - c[None, :, :]).max(axis=2)
    P = int(np.triu(cheb == 1, k=1).sum())
    assert total == g.n + 2 * P


# ---------------------------------------------------------------------------
# Decode and block metadata
# ---------------------------------------------------------------------------

LOG2WS = [6, 7, 8, 9]


def _leaf_masks(coords_in_order, leaf_of, n_leaves):
    masks = np.zeros((n_leaves, 8, 8, 8), dtype=bool)
    o = coords_in_order.astype(np.int64)
    loc = o - (o // 8) * 8
    masks[leaf_of[1:], loc[:, 0], loc[:, 1], loc[:, 2]] = True
    return masks


@pytest.mark.parametrize("log2w", LOG2WS)
def test_decode_is_inverse_of_assignment(grid, log2w):
    _, _, g, d = grid
    W = 1 << log2w
    li, vo = g.decode(log2w)
    leaf_of, origins = g.leaves()
    nb = g.n_blocks(log2w)
    assert len(li) == nb * W
    # sentinels: exactly nBlocks*W - N of them, all at the end (last block only)
    sent = li == oracle.SENTINEL_LEAF
    assert sent.sum() == nb * W - g.n
    assert (sent == (np.arange(nb * W) >= g.n)).all()
    assert (vo[sent] == oracle.SENTINEL_OFFSET).all()
    assert nb * W - g.n < W
    # (leaf, offset) -> coordinate -> index gives back the slot's index
    L = li[~sent].astype(np.int64)
    off = vo[~sent].astype(np.int64)
    pts = origins[L].astype(np.int64) + np.stack([off // 64, (off // 8) % 8, off % 8], axis=1)
    np.testing.assert_array_equal(d.lookup(pts), np.arange(1, g.n + 1))


def test_leaves_are_contiguous_and_counted(grid):
    _, coords, g, d = grid
    leaf_of, origins = g.leaves()
    distinct = np.unique(np.floor_divide(coords.astype(np.int64), 8), axis=0)
    assert len(origins) == len(distinct)
    assert (np.diff(leaf_of[1:].astype(np.int64)) >= 0).all()
    # every leaf's origin is 8-aligned and its voxels lie in it
    assert (origins % 8 == 0).all()
    o = g.coords().astype(np.int64)
    np.testing.assert_array_equal(origins[leaf_of[1:]], (o // 8) * 8)


@pytest.mark.parametrize("log2w", LOG2WS)
def test_decode_offset_is_select_in_leaf_mask(grid, log2w):
    """voxelOffset is the r-th set bit (x-major bit order) of the leaf's 512-bit
    mask, r = index - (first index of the leaf)."""
    _, _, g, d = grid
    li, vo = g.decode(log2w)
    leaf_of, origins = g.leaves()
    masks = _leaf_masks(g.coords(), leaf_of, len(origins)).reshape(len(origins), 512)
    first = np.searchsorted(leaf_of[1:], np.arange(len(origins))) + 1
    for slot in range(g.n):
        index = slot + 1
        L = li[slot]
        r = index - first[L]
        assert vo[slot] == np.flatnonzero(masks[L])[r]


@pytest.mark.parametrize("log2w", LOG2WS)
def test_block_metadata_rank_and_invariants(grid, log2w):
    _, _, g, d = grid
    W = 1 << log2w
    fl, jm = g.blocks(log2w)
    li, _ = g.decode(log2w)
    leaf_of, origins = g.leaves()
    nl = len(origins)
    nb = g.n_blocks(log2w)
    starts = np.zeros(g.n + 2, dtype=bool)  # starts[i]: index i is the first of its leaf
    starts[1] = True
    starts[2:g.n + 1] = leaf_of[2:] != leaf_of[1:-1]
    bits = np.unpackbits(jm.view(np.uint8).reshape(nb, -1), axis=1, bitorder="little").astype(bool)
    assert not bits[:, 0].any()
    popc = bits.sum(axis=1)
    # rank: the leaf of slot s is firstLeafID + popcount(jumpMap bits 0..s)
    for b in range(nb):
        ranks = fl[b] + np.cumsum(bits[b])
        valid = min(W, g.n - b * W)
        np.testing.assert_array_equal(ranks[:valid], li[b * W:b * W + valid])
    # spans and chaining
    block_start_is_leaf_start = np.array([starts[1 + b * W] for b in range(nb)])
    assert popc.sum() == (nl - 1) - block_start_is_leaf_start[1:].sum()
    for b in range(nb - 1):
        assert fl[b + 1] == fl[b] + popc[b] + int(block_start_is_leaf_start[b + 1])


# ---------------------------------------------------------------------------
# The pages' workload
# ---------------------------------------------------------------------------

@pytest.mark.slow
def test_pages_shell_counts():
    """158 <= |p| <= 162 reproduces the shell the pages measure on."""
    want = _golden("pages_shell.txt")
    g = oracle.OracleGrid(synth.WORKLOADS["S160"]())
    _, origins = g.leaves()
    v, tol = want["active_voxels_millions"]
    assert abs(g.n / 1e6 - v) <= tol
    assert len(origins) == int(want["leaves"][0])
    v, tol = want["mean_leaf_occupancy"]
    assert abs(g.n / len(origins) - v) <= tol
