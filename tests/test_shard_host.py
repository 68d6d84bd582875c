"""Block-range shards on the CPU: the plan (vbm_shard_blocks, vbm_shard_halo on
host-only grids) against the oracle's taps, and the halo exchange itself on
world-size 2 and 3 gloo ranks.  The row packing and placing are done here with
numpy (the library's gather/scatter kernels need a GPU; tests/test_gpu_shard.py
runs them); the rows cross ranks through sparse_voxel_grid_gb300.shard's
all_to_all, exactly as on the GPU path with gloo."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

import oracle
import sparse_voxel_grid_gb300 as vbm
import synth
from sparse_voxel_grid_gb300 import shard
from tests.test_oracle_pins import GRIDS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _host_grid(coords, log2w):
    return vbm.vbm_build(coords, log2w, flags=vbm.BUILD_HOST_ONLY)


@pytest.mark.parametrize("name", sorted(GRIDS))
@pytest.mark.parametrize("log2w", [6, 9])
@pytest.mark.parametrize("world", [1, 2, 3, 5])
def test_plan_covers_every_tap(name, log2w, world):
    coords = GRIDS[name]()
    o = oracle.OracleGrid(coords)
    g = _host_grid(coords, log2w)
    info = g.info
    bb = shard.shard_blocks(g, world)
    assert bb[0] == 0 and bb[-1] == info["n_blocks"] and (np.diff(bb.astype(np.int64)) >= 0).all()
    taps = o.taps(27)
    cross = o.taps(7)
    W = 1 << log2w
    covered = np.zeros(o.n + 1, dtype=np.int64)
    for q in range(world):
        b0, b1 = int(bb[q]), int(bb[q + 1])
        lo, hi = 1 + b0 * W, min(o.n, b1 * W)
        halo = shard.shard_halo(g, b0, b1)
        assert (np.diff(halo.astype(np.int64)) > 0).all()  # sorted, no repeats
        assert ((halo < lo) | (halo > hi)).all() and ((halo >= 1) & (halo <= o.n)).all()
        if b0 == b1:
            assert len(halo) == 0
            continue
        covered[lo:hi + 1] += 1
        need = np.union1d(taps[lo:hi + 1].ravel(), cross[lo:hi + 1].ravel())
        need = need[(need != 0) & ((need < lo) | (need > hi))]
        assert np.isin(need, halo).all(), f"shard {q}: taps outside own rows and halo"
    assert (covered[1:] == 1).all()  # the shards partition the indices


def test_halo_errors():
    g = _host_grid(GRIDS["tiny_shell"](), 7)
    lib = vbm.load()
    import ctypes
    cnt = ctypes.c_uint64(0)
    nb = g.info["n_blocks"]
    assert lib.vbm_shard_halo(g.handle, 2, 1, None, 0, ctypes.byref(cnt)) == -1
    assert lib.vbm_shard_halo(g.handle, 0, nb + 1, None, 0, ctypes.byref(cnt)) == -1
    assert lib.vbm_shard_halo(g.handle, 0, 1, None, 0, None) == -1
    assert lib.vbm_shard_halo(g.handle, 0, 1, None, 0, ctypes.byref(cnt)) == 0 and cnt.value > 0
    buf = (ctypes.c_uint32 * 1)()
    assert lib.vbm_shard_halo(g.handle, 0, 1, buf, 1, ctypes.byref(cnt)) == -3
    assert lib.vbm_shard_blocks(g.handle, 0, buf) == -1


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _exchange_rank(rank, world, port, workload, log2w, C, q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import oracle as orc
    import sparse_voxel_grid_gb300 as v
    import synth as syn
    from sparse_voxel_grid_gb300 import shard as sh
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        coords = syn.WORKLOADS[workload]()
        g = v.vbm_build(coords, log2w, flags=v.BUILD_HOST_ONLY)
        plan = sh.ShardPlan(g, world, rank)
        full = syn.sidecar_uniform(g.n, C, seed=11).reshape(-1, C)
        local = np.full_like(full, np.nan)
        lo, hi = plan.lo[rank], plan.hi[rank]
        local[lo:hi + 1] = full[lo:hi + 1]  # this rank's own rows only
        sendbuf = torch.from_numpy(np.ascontiguousarray(local[plan.send_order().astype(np.int64)]).ravel())
        recv = sh.exchange_packed(plan, sendbuf, C).numpy().reshape(-1, C)
        local[plan.recv_order().astype(np.int64)] = recv
        # every tap row of every own voxel is now defined and equal to the global row
        taps = orc.OracleGrid(coords).taps(27)[lo:hi + 1].ravel()
        taps = taps[taps != 0].astype(np.int64)
        ok = bool(np.array_equal(local[taps].view(np.uint32), full[taps].view(np.uint32)))
        q.put((rank, ok, len(plan.halo[rank])))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("workload,log2w,world,C", [("T", 6, 2, 3), ("T", 7, 3, 1), ("S185", 9, 2, 4)])
def test_halo_exchange_gloo(workload, log2w, world, C):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_exchange_rank, args=(r, world, port, workload, log2w, C, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = {}
    for _ in procs:
        rank, ok, nh = q.get(timeout=300)
        got[rank] = (ok, nh)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert all(ok for ok, _ in got.values()), got
    assert all(nh > 0 for _, nh in got.values())


def test_more_shards_than_blocks_and_empty_grids():
    """Shards beyond the number of blocks are empty (no blocks, no halo) and
    the non-empty ones still partition the indices; an empty grid gives empty
    shards."""
    coords = GRIDS["tiny_shell"]()
    g = _host_grid(coords, 9)
    nb = g.info["n_blocks"]
    world = nb + 3
    bb = shard.shard_blocks(g, world)
    assert bb[0] == 0 and bb[-1] == nb
    sizes = np.diff(bb.astype(np.int64))
    assert (sizes >= 0).all() and sizes.sum() == nb and (sizes == 0).sum() == world - nb
    for q in range(world):
        h = shard.shard_halo(g, int(bb[q]), int(bb[q + 1]))
        assert (len(h) == 0) == (sizes[q] == 0)
    plan = shard.ShardPlan(g, world, world - 1)
    assert sum(len(x) for x in plan.recv_rows) == len(plan.halo[world - 1])
    e = _host_grid(np.zeros((0, 3), dtype=np.int32), 7)
    assert (shard.shard_blocks(e, 4) == 0).all()
    assert len(shard.shard_halo(e, 0, 0)) == 0


def test_row_calls_validate_on_the_host():
    """vbm_gather_rows / vbm_scatter_rows reject a bad channel count and
    unaligned or NULL pointers before any CUDA call, and do nothing for a zero
    count."""
    import ctypes
    lib = vbm.load()
    P = ctypes.c_void_p
    assert lib.vbm_gather_rows(P(16), 0, P(16), 1, P(16), None) == -1
    assert lib.vbm_scatter_rows(P(16), 65, P(16), 1, P(16), None) == -1
    assert lib.vbm_gather_rows(P(16), 1, P(16), 0, P(16), None) == 0  # nothing to move
    assert lib.vbm_gather_rows(None, 1, P(16), 1, P(16), None) == -1
    assert lib.vbm_scatter_rows(P(18), 1, P(16), 1, P(16), None) == -6
