"""The oracle's box filter of every voxel of a full-size workload, on all host
cores: the index range is cut into one slice per core, and each slice is
filtered by the unmodified single-threaded oracle in a spawned process (spawned,
not forked: the test process holds a CUDA context).  Each worker rebuilds the
workload and its sidecars from the same seeded generators, so only the
slices' outputs cross process boundaries."""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np


def _sidecar(kind: str, n: int, C: int, seed: int) -> np.ndarray:
    import synth
    return synth.sidecar_uniform(n, C, seed=seed) if kind == "uniform" else synth.sidecar_normal(n, C, seed=seed)


def _box_slice(task):
    workload, kind, widths, seeds, lo, hi = task
    import oracle
    import synth

    o = oracle.OracleGrid(synth.WORKLOADS[workload]())
    which = np.arange(lo, hi, dtype=np.int64)
    return lo, [o.box_filter(_sidecar(kind, o.n, C, s), C, which=which) for C, s in zip(widths, seeds)]


def box_filter_all(workload: str, n: int, widths, seeds, kind: str = "uniform", procs: int | None = None,
                   timeout: float = 900.0):
    """Oracle box filter of rows 0..n of each sidecar (widths[i] channels, seed
    seeds[i], U[-1,1) or N(0,1) by `kind`) of `workload`; row 0 is +0.0.
    Returns one (n+1)*C float32 array per width.  Raises
    multiprocessing.TimeoutError after `timeout` seconds (a worker that died
    is replaced by the pool, and its slice would never arrive)."""
    procs = max(1, min(procs or os.cpu_count() or 1, n))
    bounds = np.linspace(1, n + 1, procs + 1).astype(np.int64)
    tasks = [(workload, kind, tuple(widths), tuple(seeds), int(bounds[i]), int(bounds[i + 1]))
             for i in range(procs) if bounds[i] < bounds[i + 1]]
    full = [np.zeros((n + 1) * C, dtype=np.float32) for C in widths]
    with mp.get_context("spawn").Pool(len(tasks)) as pool:
        for lo, outs in pool.map_async(_box_slice, tasks).get(timeout=timeout):
            for k, C in enumerate(widths):
                full[k][lo * C: lo * C + len(outs[k])] = outs[k]
    return full
