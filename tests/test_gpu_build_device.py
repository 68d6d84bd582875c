"""vbm_build_device (GPU builder) against vbm_build (host builder): every
exported array and every statistic must be identical, on small grids, the
full workloads and the error cases."""
import numpy as np
import pytest

import sparse_voxel_grid_gb300 as vbm
import synth
from tests import gpu_util as gu
from tests.test_oracle_pins import GRIDS

pytestmark = pytest.mark.gpu

ARRAYS = ["leaf_mask", "leaf_prefix", "leaf_first", "leaf_origin", "block_first_leaf", "block_jump",
          "leaf_neighbours"]
STATS = ["n_active", "n_leaves", "n_blocks", "block_width", "n_upper", "n_lower", "n_blocks_over_cache",
         "max_span", "device_bytes"]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    gu.require_gpu()


def _same(coords, log2w, flags=0):
    t = gu.torch()
    h = vbm.vbm_build(coords, log2w, flags)
    d = vbm.vbm_build_device(t.from_numpy(np.ascontiguousarray(coords, dtype=np.int32)).cuda(), log2w, flags)
    for k in STATS:
        assert h.info[k] == d.info[k], k
    for a in ARRAYS:
        np.testing.assert_array_equal(vbm.vbm_leaf_export(d, a), vbm.vbm_leaf_export(h, a), err_msg=a)
    return h, d


SMALL = {k: v for k, v in GRIDS.items() if k != "clusters"}  # clusters reach 2,000,000 (> 2^20)
SMALL["scatter"] = lambda: synth.scatter(side=10, count=700, origin=-37, seed=5)
SMALL["near_limit"] = lambda: np.array([[2 ** 20 - 1, -(2 ** 20) + 1, 5], [-8, 7, 0], [2 ** 20 - 9, 0, 0]],
                                       dtype=np.int32)


@pytest.mark.parametrize("name", sorted(SMALL))
@pytest.mark.parametrize("log2w", [6, 9])
def test_small_grids_identical(name, log2w):
    _same(SMALL[name](), log2w)


@pytest.mark.parametrize("name,log2w", [("S185", 7), ("S185", 9), ("D", 8), ("F", 8)])
def test_workloads_identical(name, log2w):
    h, d = _same(synth.WORKLOADS[name](), log2w)
    # the filters on the two grids agree bit for bit
    t = gu.torch()
    C = 3
    s = gu.to_dev(synth.sidecar_uniform(h.n, C, seed=1))
    a = gu.box_filter(h, s, C, vbm.RESOLVE_BRICK, vbm.OUTPUT_STREAMED)
    b = gu.box_filter(d, s, C, vbm.RESOLVE_BRICK, vbm.OUTPUT_STREAMED)
    np.testing.assert_array_equal(gu.bits(a), gu.bits(b))
    del t


def test_one_voxel_per_leaf_takes_the_large_table():
    # 100,000 voxels in 100,000 leaves: more leaves than the first hash table
    # (sized for one leaf per 16 voxels) holds, so the build retries with the
    # table of 2n slots
    c = synth.scatter(side=47, count=100_000, origin=-200, seed=9)
    assert len(c) == 100_000
    h, d = _same(c, 7)
    assert d.info["n_leaves"] == 100_000


def test_duplicates_and_dedup():
    t = gu.torch()
    c = np.array([[0, 0, 0], [1, 2, 3], [0, 0, 0], [9, 9, 9], [1, 2, 3]], dtype=np.int32)
    with pytest.raises(vbm.VbmError) as e:
        vbm.vbm_build_device(t.from_numpy(c).cuda(), 7)
    assert e.value.code == -2
    _same(c, 7, vbm.BUILD_DEDUP)


def test_range_and_empty():
    t = gu.torch()
    c = np.array([[2 ** 20, 0, 0]], dtype=np.int32)
    with pytest.raises(vbm.VbmError) as e:
        vbm.vbm_build_device(t.from_numpy(c).cuda(), 7)
    assert e.value.code == -3
    g = vbm.vbm_build_device(t.zeros((0, 3), dtype=t.int32, device="cuda"), 7)
    assert g.n == 0 and g.info["n_blocks"] == 0
