"""Benchmark of the sparse voxel-grid stencil pipeline on one GB300.

Workload: the sphere shell of radius 185 and thickness 3 (183.5 <= |p| <= 186.5,
1,290,538 active voxels in 11,255 leaves), fp32 sidecars U[-1,1) with C
interleaved channels.  One step = the 27-tap box filter (select-based decode +
brick resolver + streamed gather/accumulate, fused) over every active voxel of
four sidecars, C = 1, 3, 8 and 16, BlockWidth 512, in one
vbm_box_filter_batch call: one launch in which each CTA decodes one VBM block,
builds its index bricks once and runs all four sidecars' gathers from them
(`--step separate`: four calls).  `value` counts each voxel once per sidecar:
4 * N voxels per step.  Each width is also timed alone (`detail`); the
one-channel filters that the stated target names (the pages' cached streamed
resolver at W = 128 and 512, and the brick resolver) are timed against the
least time of a kernel with their launch shape (`target`); the other
resolvers (the pages' tree walk and cached table), both output modes, both
block widths, the cross Laplacian, the WENO consumer, the decodes and the
builders are timed in `variants`.

Timing: each step (and each detail launch) is bracketed by CUDA events on the
launching stream; L2 is flushed (a write of twice its size) before each,
outside the events.  A JSON line is printed on rank 0.  `--impl reference`
times the CPU oracle on the host cores instead, on a bounded sample of the
same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

CS = (1, 3, 8, 16)
LOG2W = 9
METRIC = "active voxels/s (27-tap box filter, C=1..16) and achieved HBM GB/s vs GB300 peak"
WORKLOADS = {
    "T": "T tiny sphere shell 11.5<=|p|<=13.5",
    "S185": "S185 sphere shell 183.5<=|p|<=186.5",
    "S160": "S160 sphere shell 158<=|p|<=162 (the pages' shell counts)",
    "D": "D random 8^3 bricks on [0,512)^3 (leaf p=0.3, density U[0.01,1])",
    "F": "F 4-octave value-noise fog on [0,512)^3 (> 0.55)",
}
LEAF_META_BYTES = 88  # mask 64 + 9-bit directory 8 + first index 4 + origin 12


def algorithmic_bytes(n, n_leaves, n_blocks, W, C):
    """Unique bytes a launch must move: sidecar rows read, output rows written,
    leaf metadata and block metadata (tree-node reads excluded)."""
    return 8 * C * n + 8 * C + LEAF_META_BYTES * n_leaves + (4 + W // 8) * n_blocks


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms (the caller
    keeps the GPU busy with the benchmarked step while sampling)."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons, power = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            try:
                power.append(float(f[3]))
            except ValueError:
                pass
            for name, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm),
                "power_w": statistics.median(power) if power else None}


def max_over_ranks(value: float, device=None) -> float:
    """Largest `value` over the ranks of the default process group (any
    backend); `value` itself when no group is initialised."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_gpu(args):
    import torch

    import sparse_voxel_grid_gb300 as vbm
    import synth

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    coords = synth.WORKLOADS[args.workload]()
    g = vbm.vbm_build_device(torch.from_numpy(coords).cuda(), args.log2w)
    info = g.info
    n, W = info["n_active"], info["block_width"]
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    flush_buf = torch.empty(max(2 * l2, 64 << 20) // 4, dtype=torch.float32, device="cuda")

    sidecars = {C: torch.from_numpy(synth.sidecar_uniform(n, C, seed=0)).cuda() for C in CS}
    outs = {C: torch.empty_like(sidecars[C]) for C in CS}

    resolver = {"cached": vbm.RESOLVE_CACHED, "brick": vbm.RESOLVE_BRICK, "walk": vbm.RESOLVE_TREEWALK}[args.resolver]

    def launch(C, output=vbm.OUTPUT_STREAMED, grid=g):
        vbm.vbm_box_filter(grid, sidecars[C], C, outs[C], resolver, output, stream)

    def launch_step():
        if args.step == "batch":  # all widths in one call (one launch with the brick resolver)
            vbm.vbm_box_filter_batch(g, [sidecars[C] for C in CS], list(CS), [outs[C] for C in CS], resolver, stream)
        else:
            for C in CS:
                launch(C)

    def timed_launch(fn):
        flush_buf.zero_()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        return e0, e1

    # warm-up
    for _ in range(args.warmup):
        timed_launch(launch_step)
        for C in CS:
            timed_launch(lambda C=C: launch(C))
    torch.cuda.synchronize()

    # timed region: K steps, L2 flushed before each (outside the events)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        # The same step, untimed, for ~0.6 s first, so that the 200 ms clock
        # samples see the GPU under this load (the K timed steps alone last a
        # few ms); then the K timed steps.
        busy_until = time.perf_counter() + 0.6
        while time.perf_counter() < busy_until:
            for _ in range(50):
                flush_buf.zero_()
                launch_step()
            torch.cuda.synchronize()
        t0 = time.perf_counter()
        step_evs = [timed_launch(launch_step) for _ in range(args.steps)]
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        wall = time.perf_counter() - t0
    step_ms = [a.elapsed_time(b) for a, b in step_evs]
    ms_per_step = statistics.mean(step_ms)
    if dist:
        ms_per_step = max_over_ranks(ms_per_step, device="cuda")
    value = world * len(CS) * n / (ms_per_step * 1e-3)

    # per-width detail: each width alone, K launches, L2 flushed before each
    evs = {C: [timed_launch(lambda C=C: launch(C)) for _ in range(args.steps)] for C in CS}
    torch.cuda.synchronize()
    per_c_ms = {C: [a.elapsed_time(b) for a, b in evs[C]] for C in CS}

    peak_gbs, peak_kind = peaks()
    detail = {}
    for C in CS:
        ms = statistics.mean(per_c_ms[C])
        b = algorithmic_bytes(n, info["n_leaves"], info["n_blocks"], W, C)
        detail[f"C{C}"] = {"ms_mean": round(ms, 5), "ms_median": round(statistics.median(per_c_ms[C]), 5),
                           "ms_min": round(min(per_c_ms[C]), 5), "voxels_per_s": n / (ms * 1e-3),
                           "alg_bytes": b, "gbs": b / (ms * 1e-3) / 1e9,
                           "frac_of_hbm": b / (ms * 1e-3) / 1e9 / peak_gbs}
    if args.step == "batch":  # the step's kernel is the batched launch
        dom_label = f"box filter batch ({args.resolver} resolver, C=1,3,8,16 in one call)"
        dom_ms = ms_per_step
        dom_bytes = sum(algorithmic_bytes(n, info["n_leaves"], info["n_blocks"], W, C) for C in CS)
        traffic = load_traffic(f"box_{args.resolver}_batch_W{W}")
        l1_wavefronts = load_traffic(f"box_{args.resolver}_batch_W{W}_l1_wavefronts")
    else:
        l1_wavefronts = None
        dom = max(CS, key=lambda C: statistics.mean(per_c_ms[C]))
        dom_label = f"box filter ({args.resolver} resolver, streamed) C={dom}"
        dom_ms = statistics.mean(per_c_ms[dom])
        dom_bytes = algorithmic_bytes(n, info["n_leaves"], info["n_blocks"], W, dom)
        traffic = load_traffic(f"box_{args.resolver}_W{W}_C{dom}")
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9

    target = None
    if not args.no_target:
        target = run_target(torch, vbm, coords, g, sidecars, outs, timed_launch, args, peak_gbs)

    # end to end through the public API: pinned host sidecar -> device -> filter -> host
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(torch, vbm, g, n, sidecars, outs, args, stream, resolver)

    variants = run_variants(torch, vbm, coords, sidecars, outs, timed_launch, args) if not args.no_variants else None
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(coords, sample=args.cpu_sample, workload=args.workload)

    clk = clocks.summary()
    l1 = None
    if l1_wavefronts and clk.get("sm_mhz"):
        l1 = l1_data_pipe(l1_wavefronts, dom_ms, torch.cuda.get_device_properties(local).multi_processor_count,
                          clk["sm_mhz"])
    line = {
        "metric": METRIC, "value": value, "unit": "voxels/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded)",
        "config": workload_config(args, n, info["n_leaves"], info["n_blocks"], info["n_blocks_over_cache"],
                                  info["max_span"], world),
        "wall_ms_per_step_incl_flush": wall / args.steps * 1e3,
        "roofline": {"bound": "hbm", "kernel": dom_label, "achieved": achieved,
                     "peak": peak_gbs, "unit": "GB/s", "frac": achieved / peak_gbs, "traffic": traffic,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s", "alg_bytes_per_launch": dom_bytes, "l1_data_pipe": l1},
        "detail": detail,
        "target": target,
        "e2e": e2e,
        "gpu_launches": (1 if args.step == "batch" and args.resolver == "brick" else len(CS)) * args.steps,
        "clocks": clk,
        "cpu_baseline": cpu,
        "variants": variants,
    }
    if rank == 0:
        print(json.dumps(line))
    if dist:
        dist.destroy_process_group()


def workload_config(args, n, n_leaves, n_blocks, n_over, max_span, world):
    """The `config` object both arms print for the same workload."""
    W = 1 << args.log2w
    return {"workload": f"{WORKLOADS[args.workload]}, N={n}, leaves={n_leaves}, fused decode + {args.resolver} "
                        f"resolver + streamed 27-tap box filter at C=1,3,8,16, W={W}",
            "step": "one vbm_box_filter_batch call (one launch with the brick resolver)" if args.step == "batch"
                    else "four vbm_box_filter calls",
            "n_active": n, "n_leaves": n_leaves, "block_width": W, "channels": list(CS), "n_blocks": n_blocks,
            "n_blocks_over_cache": n_over, "max_span": max_span, "resolver": args.resolver, "output": "streamed",
            "l2": "flushed before every launch", "value_counts": "4*N voxels per step (one per channel width)",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def l1_data_pipe(wavefronts, ms, sms, sm_mhz):
    """The batched kernel's real bound: L1 data-pipe wavefronts per launch
    (the committed ncu count) over the live launch time, against one wavefront
    per SM per clock at the sampled SM clock."""
    cap = ms * 1e-3 * sms * sm_mhz * 1e6
    return {"wavefronts_per_launch": wavefronts, "peak": "1 wavefront / SM / clock", "frac": wavefronts / cap}


def load_traffic(key):
    """DRAM bytes per launch from the committed ncu summary, if it covers `key`
    and the kernel sources are unchanged since the counters were taken."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    h = hashlib.sha1()
    for f in d.get("source_files", []):
        fp = os.path.join(ROOT, f)
        if not os.path.exists(fp):
            return None
        h.update(open(fp, "rb").read())
    if h.hexdigest() != d.get("source_sha1"):
        return None
    return d.get(key)


def run_target(torch, vbm, coords, g512, sidecars, outs, timed_launch, args, peak_gbs):
    """The stated target: the fused cached box filter at C=1 on the shell at
    >= 60% of the HBM roofline.  Times the one-channel box filters it concerns
    (the pages' cached streamed resolver at W = 128 and 512, and the brick
    resolver at both widths) and, beside them, the probe kernels with the same
    launch shape: an empty kernel (the least time any kernel of that shape
    takes after an L2 flush), one that only loads each block's metadata, and
    one that only follows the brick resolver's chain of dependent loads.
    Median of --steps launches each, L2 flushed before every launch."""
    reps = max(args.steps, 10)

    def tmed(fn):
        for _ in range(3):
            timed_launch(fn)
        evs = [timed_launch(fn) for _ in range(reps)]
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in evs)

    grids = {512: g512}
    if g512.info["block_width"] != 128:
        grids[128] = vbm.vbm_build_device(torch.from_numpy(coords).cuda(), 7)
    s1, o1 = sidecars[1], outs[1]
    rows, floors = [], {}
    for W in sorted(grids):
        g = grids[W]
        info = g.info
        b = algorithmic_bytes(info["n_active"], info["n_leaves"], info["n_blocks"], W, 1)
        for name, resolver in (("cached streamed", vbm.RESOLVE_CACHED), ("brick", vbm.RESOLVE_BRICK)):
            ms = tmed(lambda: vbm.vbm_box_filter(g, s1, 1, o1, resolver, vbm.OUTPUT_STREAMED))
            key = f"box_{name.split()[0]}_W{W}_C1"
            rows.append({"kernel": f"box filter C=1, {name}", "W": W, "ms": round(ms, 5), "alg_bytes": b,
                         "gbs": b / (ms * 1e-3) / 1e9, "frac": b / (ms * 1e-3) / 1e9 / peak_gbs,
                         "thread_inst_per_voxel": load_traffic(key + "_thread_inst_per_voxel"),
                         "dram_bytes": load_traffic(key)})
        fl = {}
        for kname, kind in (("empty", vbm.PROBE_EMPTY), ("metadata", vbm.PROBE_METADATA),
                            ("chain", vbm.PROBE_CHAIN)):
            fl[f"{kname}_ms"] = round(tmed(lambda: vbm.vbm_probe_launch(g, kind, s1)), 5)
        fl["ctas"] = info["n_blocks"]
        fl["frac_if_kernel_took_empty_ms"] = b / (fl["empty_ms"] * 1e-3) / 1e9 / peak_gbs
        floors[f"W{W}"] = fl
    for W, g in grids.items():
        if g is not g512:
            g.close()
    return {"statement": "fused cached box filter, C=1, on the ~1.3M-voxel shell at >= 60% of the HBM roofline",
            "peak_gbs": peak_gbs, "kernels": rows, "launch_floor": floors,
            "how": "median of the event times of repeated launches, L2 flushed before each; alg_bytes as the "
                   "headline (sidecar read + output write + leaf and block metadata); launch_floor: probe "
                   "kernels of the same launch shape (include/vbm_probe.h)"}


def run_e2e(torch, vbm, g, n, sidecars, outs, args, stream, resolver):
    """The step through the library's host-buffer call: every step is one
    vbm_box_filter_batch_host call on pinned host sidecars (copies in, the
    batched filter, copies back, all inside the call; consecutive calls
    overlap on the grid's staging sets); wall clock over K steps.  Beside it,
    the host link's own copy rate for the same bytes (each direction alone,
    then both at once), which bounds it."""
    host_in = [sidecars[C].cpu().pin_memory() for C in CS]
    host_out = [torch.empty_like(h).pin_memory() for h in host_in]

    def step():
        vbm.vbm_box_filter_batch_host(g, host_in, list(CS), host_out, resolver, stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    ms = (time.perf_counter() - t0) * 1e3 / args.steps
    for C, h in zip(CS, host_out):  # the copies really carried the filter outputs
        assert torch.equal(h, outs[C].cpu()), "e2e output differs from the device-timed output"
    bi = sum(h.numel() * 4 for h in host_in)
    bo = sum(h.numel() * 4 for h in host_out)
    return {"value": len(CS) * n / (ms * 1e-3), "unit": "voxels/s", "ms_per_step": ms,
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "link": host_link(torch, bi, args.steps),
            "how": "one vbm_box_filter_batch_host call per step (pinned host sidecars -> device -> batched box "
                   "filter -> pinned host outputs, inside the library); wall clock over K steps"}


def host_link(torch, nbytes, reps):
    """Copy rate of the host link for `nbytes` each way (pinned host memory,
    one cudaMemcpyAsync per direction per repetition): host to device alone,
    device to host alone, and both at once on two streams; the best of three
    timings of `reps` copies each.  GB/s."""
    h_in = torch.empty(nbytes // 4, dtype=torch.float32).pin_memory()
    h_out = torch.empty_like(h_in).pin_memory()
    d_in = torch.empty(nbytes // 4, dtype=torch.float32, device="cuda")
    d_out = torch.empty_like(d_in)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def rate(h2d, d2h):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(reps):
            if h2d:
                with torch.cuda.stream(s1):
                    d_in.copy_(h_in, non_blocking=True)
            if d2h:
                with torch.cuda.stream(s2):
                    h_out.copy_(d_out, non_blocking=True)
        torch.cuda.synchronize()
        return (h2d + d2h) * nbytes * reps / (time.perf_counter() - t0) / 1e9

    rate(True, True)
    best = lambda h2d, d2h: max(rate(h2d, d2h) for _ in range(3))  # noqa: E731 (best of three: the link's capacity)
    return {"h2d_gbs": best(True, False), "d2h_gbs": best(False, True), "both_gbs": best(True, True),
            "bytes_each_way": nbytes, "how": "best of three repetitions per direction"}


def run_variants(torch, vbm, coords, sidecars, outs, timed_launch, args):
    """Every box variant (resolver x output x W x C), the cross Laplacian and
    the decode on the shell, each timed cold-cache (mean of a few launches)."""
    reps = args.variant_reps
    res = []

    def tmean(fn):
        for _ in range(2):
            timed_launch(fn)
        evs = [timed_launch(fn) for _ in range(reps)]
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) for a, b in evs)

    for log2w in (7, 9):
        g = vbm.vbm_build(coords, log2w)
        for C in CS:
            for rname, r in (("walk", vbm.RESOLVE_TREEWALK), ("cached", vbm.RESOLVE_CACHED),
                             ("brick", vbm.RESOLVE_BRICK)):
                outputs = (("streamed", vbm.OUTPUT_STREAMED), ("materialised", vbm.OUTPUT_MATERIALISED))
                for oname, o in (outputs if r != vbm.RESOLVE_BRICK else outputs[:1]):
                    ms = tmean(lambda: vbm.vbm_box_filter(g, sidecars[C], C, outs[C], r, o))
                    res.append({"kernel": "box", "W": 1 << log2w, "C": C, "resolver": rname, "output": oname,
                                "ms": round(ms, 5)})
        g.close()
    # grid builders (host C++ and GPU), wall time including upload / allocation
    dcoords = torch.from_numpy(coords).cuda()
    for name, fn in (("build_host", lambda: vbm.vbm_build(coords, 9)),
                     ("build_device", lambda: vbm.vbm_build_device(dcoords, 9))):
        fn().close()
        ts = []
        for _ in range(3):
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            g = fn()
            torch.cuda.synchronize()
            ts.append(time.perf_counter() - t0)
            g.close()
        res.append({"kernel": name, "W": 512, "ms": round(1e3 * statistics.median(ts), 3)})
    for log2w in (6, 7, 8, 9):
        g = vbm.vbm_build(coords, log2w)
        for rname, r in (("walk", vbm.RESOLVE_TREEWALK), ("cached", vbm.RESOLVE_CACHED),
                         ("brick", vbm.RESOLVE_BRICK)):
            ms = tmean(lambda: vbm.vbm_cross_filter(g, sidecars[1], 1, outs[1], r, vbm.CROSS_LAPLACIAN))
            res.append({"kernel": "laplacian", "W": 1 << log2w, "C": 1, "resolver": rname, "ms": round(ms, 5)})
            ms = tmean(lambda: vbm.vbm_weno_filter(g, sidecars[1], outs[1], 0.0, r))
            res.append({"kernel": "weno", "W": 1 << log2w, "C": 1, "resolver": rname, "ms": round(ms, 5)})
        li = torch.empty(g.n_slots, dtype=torch.int32, device="cuda")
        vo = torch.empty(g.n_slots, dtype=torch.int16, device="cuda")
        for mname, fn in (("select", vbm.vbm_decode), ("sweep", vbm.vbm_decode_sweep)):
            ms = tmean(lambda: fn(g, li, vo))
            res.append({"kernel": "decode", "method": mname, "W": 1 << log2w, "ms": round(ms, 5)})
        g.close()
    return res


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------

def _oracle_box_worker(task):
    """One host process of the all-cores oracle timing: the box filter of
    voxels [lo, hi) of the workload at every channel width, compute time only."""
    workload, lo, hi = task
    import oracle
    import synth

    o = oracle.OracleGrid(synth.WORKLOADS[workload]())
    sides = {C: synth.sidecar_uniform(o.n, C, seed=0) for C in CS}
    which = np.arange(lo, hi, dtype=np.int64)
    t0 = time.perf_counter()
    for C in CS:
        o.box_filter(sides[C], C, which=which)
    return time.perf_counter() - t0


def cpu_baseline(coords, sample, workload="S185", procs=None, per_process=100_000):
    """The oracle, as it stands, on the host cores.

    - Single process: the stages timed separately (index build, decode of
      every slot, box filter at each C and the Laplacian on a sample).
    - All cores: the unmodified single-threaded oracle in one spawned process
      per core, each filtering a disjoint slice of the first
      min(N, cores * per_process) voxels; the value counts the voxels of all
      slices over the slowest process's compute time.
    """
    import multiprocessing as mp

    import oracle
    import synth

    t0 = time.perf_counter()
    o = oracle.OracleGrid(coords)
    t_build = time.perf_counter() - t0
    t0 = time.perf_counter()
    o.decode(LOG2W)
    t_decode = time.perf_counter() - t0
    which = np.arange(1, min(sample, o.n) + 1, dtype=np.int64)
    t = 0.0
    stages = {"index_build_s": round(t_build, 3), "decode_all_slots_s": round(t_decode, 3)}
    for C in CS:
        s = synth.sidecar_uniform(o.n, C, seed=0)
        t0 = time.perf_counter()
        o.box_filter(s, C, which=which)
        dt = time.perf_counter() - t0
        stages[f"box_C{C}_voxels_per_s"] = round(len(which) / dt)
        t += dt
    s1 = synth.sidecar_uniform(o.n, 1, seed=0)
    t0 = time.perf_counter()
    o.cross_filter(s1, 1, op=0, which=which)
    stages["laplacian_voxels_per_s"] = round(len(which) / (time.perf_counter() - t0))
    single = len(CS) * len(which) / t

    procs = procs or max(1, os.cpu_count() or 1)
    # each process holds the whole grid and its sidecars (~160 B per voxel):
    # keep the total under ~24 GB of host memory
    procs = max(1, min(procs, int(24e9 // max(1, 160 * o.n))))
    m = min(o.n, procs * per_process)
    per = -(-m // procs)
    tasks = [(workload, 1 + i * per, min(m, (i + 1) * per) + 1) for i in range(procs) if 1 + i * per <= m]
    with mp.get_context("spawn").Pool(len(tasks)) as pool:
        times = pool.map_async(_oracle_box_worker, tasks).get(timeout=600)
    all_cores = len(CS) * m / max(times)
    return {"value": all_cores, "unit": "voxels/s", "cores": len(tasks), "kind": "oracle",
            "sample": f"the first {m} of {o.n} voxels at C=1,3,8,16, split into {len(tasks)} slices, one "
                      f"spawned process per core running the single-threaded C++ oracle (index build and "
                      f"sidecar generation in each process not counted)",
            "seconds": max(times),
            "single_core": {"value": single, "cores": 1,
                            "sample": f"first {len(which)} voxels at C=1,3,8,16", "seconds": t},
            "stages_single_core": stages}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    import synth

    coords = synth.WORKLOADS[args.workload]()
    o = oracle.OracleGrid(coords)
    sides = {C: synth.sidecar_uniform(o.n, C, seed=0) for C in CS}
    # Size the per-step sample so that warm-up + timed steps take about
    # --reference-seconds in total (calibrated on 2000 voxels).
    probe = np.arange(1, min(2000, o.n) + 1, dtype=np.int64)
    t0 = time.perf_counter()
    for C in CS:
        o.box_filter(sides[C], C, which=probe)
    per_voxel = (time.perf_counter() - t0) / len(probe)
    budget = args.reference_seconds / max(1, args.steps + args.warmup)
    m = int(min(args.cpu_sample, o.n, max(2000, budget / per_voxel)))
    which = np.arange(1, m + 1, dtype=np.int64)

    def step():
        for C in CS:
            o.box_filter(sides[C], C, which=which)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = len(CS) * len(which) / dt
    sample = f"first {len(which)} of {o.n} voxels per step, C=1,3,8,16 (single-threaded C++ oracle)"
    _, origins = o.leaves()
    fl, jm = o.blocks(args.log2w)
    spans = 1 + np.array([sum(bin(int(w)).count("1") for w in row) for row in jm], dtype=np.int64)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "voxels/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded)",
        "config": {**workload_config(args, o.n, len(origins), len(fl), int((spans > 16).sum()),
                                     int(spans.max()) if len(spans) else 0, world),
                   "sample_voxels": len(which)},
        "cpu_baseline": {"value": value, "unit": "voxels/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "voxels/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def run_decode_ab(args):
    """Select decode against the sweep decode it replaced, on the shells and
    the decode grid D at every block width: median of --steps cold-cache
    launches each (L2 flushed before every launch), outputs compared byte for
    byte.  Prints one JSON line."""
    import torch
    import sparse_voxel_grid_gb300 as vbm
    import synth

    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    flush_buf = torch.empty(max(2 * l2, 64 << 20) // 4, dtype=torch.float32, device="cuda")

    def median_us(fn):
        for _ in range(args.warmup):
            fn()
        evs = []
        for _ in range(args.steps):
            flush_buf.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in evs) * 1e3

    rows = []
    for name in ("S185", "S160", "D"):
        coords = torch.from_numpy(synth.WORKLOADS[name]()).cuda()
        for log2w in (6, 7, 8, 9):
            g = vbm.vbm_build_device(coords, log2w)
            m = g.n_slots
            maps = {}
            for mname, fn in (("select", vbm.vbm_decode), ("sweep", vbm.vbm_decode_sweep)):
                li = torch.full((m,), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
                vo = torch.full((m,), 0x5555, dtype=torch.int16, device="cuda")
                maps[mname] = (li, vo, median_us(lambda: fn(g, li, vo)))
            same = bool(torch.equal(maps["select"][0], maps["sweep"][0]) and
                        torch.equal(maps["select"][1], maps["sweep"][1]))
            sel, swp = maps["select"][2], maps["sweep"][2]
            rows.append({"workload": name, "n": g.n, "leaves": g.info["n_leaves"], "W": 1 << log2w,
                         "select_us": round(sel, 2), "sweep_us": round(swp, 2), "speedup": round(swp / sel, 3),
                         "identical": same})
            g.close()
        del coords
    print(json.dumps({"metric": "decode: select vs sweep", "unit": "us (median, L2 flushed)", "steps": args.steps,
                      "warmup": args.warmup, "rows": rows}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--resolver", choices=["cached", "brick", "walk"], default="brick")
    ap.add_argument("--log2w", type=int, default=LOG2W, choices=[6, 7, 8, 9])
    ap.add_argument("--workload", default="S185", choices=sorted(WORKLOADS),
                    help="input grid (default: the S185 shell, the headline workload)")
    ap.add_argument("--cpu-sample", type=int, default=150000)
    ap.add_argument("--reference-seconds", type=float, default=90.0)
    ap.add_argument("--variant-reps", type=int, default=5)
    ap.add_argument("--no-variants", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-target", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--step", choices=["batch", "separate"], default="batch",
                    help="the four widths in one vbm_box_filter_batch call (default) or four calls")
    ap.add_argument("--decode-ab", action="store_true",
                    help="time the select decode against the sweep decode and print that table instead")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "gb300":
        args.warmup = 3
    if args.decode_ab:
        run_decode_ab(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
