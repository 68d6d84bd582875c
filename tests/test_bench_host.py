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


def test_l1_data_pipe_fraction():
    # 56.08M wavefronts in 0.2109 ms on 152 SMs at 2,070 MHz: 0.845 of one per SM per clock
    r = bench.l1_data_pipe(56083773, 0.2109136, 152, 2070.0)
    assert abs(r["frac"] - 56083773 / (0.2109136e-3 * 152 * 2070e6)) < 1e-12
    assert 0.84 < r["frac"] < 0.85


def test_traffic_is_dropped_when_sources_change(tmp_path, monkeypatch):
    import json
    src = tmp_path / "k.cu"
    src.write_text("kernel v1")
    (tmp_path / "profiles").mkdir()
    import hashlib
    h = hashlib.sha1(b"kernel v1").hexdigest()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
        {"source_files": ["k.cu"], "source_sha1": h, "box_brick_batch_W512": 123}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_traffic("box_brick_batch_W512") == 123
    src.write_text("kernel v2")
    assert bench.load_traffic("box_brick_batch_W512") is None
