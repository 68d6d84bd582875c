"""The all-cores oracle helper used by the full-size GPU tests gives exactly
the single-process oracle's outputs (slices stitched in the right places,
row 0 zero)."""
import numpy as np

import oracle
import synth
from tests import oracle_pool


def test_slices_equal_one_process():
    o = oracle.OracleGrid(synth.WORKLOADS["T"]())
    widths, seeds = (1, 3, 8), (5, 6, 7)
    got = oracle_pool.box_filter_all("T", o.n, widths, seeds, procs=3)
    for C, s, g in zip(widths, seeds, got):
        want = o.box_filter(synth.sidecar_uniform(o.n, C, seed=s), C)
        np.testing.assert_array_equal(g.view(np.uint32), want.view(np.uint32))
        assert (g[:C] == 0).all()
