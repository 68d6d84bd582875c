"""Properties the GPU parity grids are built to have, checked on the CPU."""
import numpy as np

import oracle
from tests.test_gpu_parity import _absent_edge_leaves


def test_absent_edge_leaves_has_taps_past_absent_leaves():
    """The grid holds active box taps whose z-row lies in an absent leaf: tap
    (dx,dy,dz) of a voxel on its leaf's z face (dz crossing it) and on its x or
    y face (dx or dy crossing), where the leaf across the x/y face only is
    absent but the diagonal leaf across the z face as well holds the tap."""
    coords = _absent_edge_leaves()
    o = oracle.OracleGrid(coords)
    leaves = {tuple(c) for c in (coords >> 3).tolist()}
    found = 0
    for x, y, z in coords.tolist():
        for dx in (-1, 0, 1):
            for dy in (-1, 0, 1):
                for dz in (-1, 1):
                    tx, ty, tz = x + dx, y + dy, z + dz
                    crosses_xy = (tx >> 3, ty >> 3) != (x >> 3, y >> 3)
                    crosses_z = (tz >> 3) != (z >> 3)
                    if not (crosses_xy and crosses_z) or o.index(tx, ty, tz) == 0:
                        continue
                    if (tx >> 3, ty >> 3, z >> 3) not in leaves:
                        found += 1
    assert found >= 8
