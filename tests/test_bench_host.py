"""Host-side parts of bench.py that need no GPU: the oracle timed on several
host processes (spawned, each over its own slice of the workload) and the
per-stage single-process timings."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def test_cpu_baseline_on_two_processes():
    coords = synth.WORKLOADS["T"]()
    r = bench.cpu_baseline(coords, sample=500, workload="T", procs=2, per_process=1000)
    assert r["kind"] == "oracle" and r["unit"] == "voxels/s"
    assert r["cores"] == 2 and r["value"] > 0 and np.isfinite(r["value"])
    assert "first 2000 of 3992 voxels" in r["sample"]
    assert r["single_core"]["cores"] == 1 and r["single_core"]["value"] > 0
    st = r["stages_single_core"]
    for k in ("index_build_s", "decode_all_slots_s", "box_C1_voxels_per_s", "box_C16_voxels_per_s",
              "laplacian_voxels_per_s"):
        assert k in st and st[k] >= 0


def test_workload_config_is_shared_by_both_arms():
    class A:
        log2w, workload, resolver, step = 9, "S185", "brick", "batch"
    c = bench.workload_config(A, 1290538, 11255, 2521, 0, 13, 1)
    assert c["block_width"] == 512 and c["n_blocks"] == 2521 and c["channels"] == [1, 3, 8, 16]
    assert c["workload"].startswith(bench.WORKLOADS["S185"])
