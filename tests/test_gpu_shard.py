"""Block-range shards on the GPU.  The row gather/scatter kernels against numpy
indexing; the block-range filter against the whole-grid call; and the sharded
box filter end to end: world-size 2 and 3 gloo ranks, all on the one GPU
(their kernels never wait on one another; the halo rows pass between ranks
through host memory), each filtering its own blocks after the halo exchange.
The ranks' output rows, put together, must equal the oracle bit for bit."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

import oracle
import sparse_voxel_grid_gb300 as vbm
import synth
from tests import gpu_util as gu
from tests import oracle_pool

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CS = (1, 3, 8, 16)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    gu.require_gpu()


def test_gather_scatter_rows():
    t = gu.torch()
    import ctypes
    lib = vbm.load()
    rng = np.random.default_rng(0)
    for C in (1, 3, 8, 13):
        src = rng.standard_normal((1000, C)).astype(np.float32)
        rows = rng.choice(1000, size=300, replace=False).astype(np.uint32)
        sd, rd = gu.to_dev(src.ravel()), t.from_numpy(rows.astype(np.int32)).cuda()
        packed = t.full((300 * C,), float("nan"), device="cuda")
        assert lib.vbm_gather_rows(ctypes.c_void_p(sd.data_ptr()), C, ctypes.c_void_p(rd.data_ptr()), 300,
                                   ctypes.c_void_p(packed.data_ptr()), None) == 0
        dst = t.zeros(1000 * C, device="cuda")
        assert lib.vbm_scatter_rows(ctypes.c_void_p(packed.data_ptr()), C, ctypes.c_void_p(rd.data_ptr()), 300,
                                    ctypes.c_void_p(dst.data_ptr()), None) == 0
        t.cuda.synchronize()
        np.testing.assert_array_equal(packed.cpu().numpy().reshape(-1, C), src[rows])
        want = np.zeros_like(src)
        want[rows] = src[rows]
        np.testing.assert_array_equal(dst.cpu().numpy().reshape(-1, C), want)
    assert lib.vbm_gather_rows(ctypes.c_void_p(sd.data_ptr()), 0, ctypes.c_void_p(rd.data_ptr()), 1,
                               ctypes.c_void_p(packed.data_ptr()), None) == -1


@pytest.mark.parametrize("resolver", [vbm.RESOLVE_BRICK, vbm.RESOLVE_CACHED])
def test_block_ranges_equal_whole_grid(resolver):
    """Filtering blocks [b0, b1) for consecutive ranges that cover the grid
    writes exactly the whole-grid call's outputs; rows outside a range are
    left untouched."""
    t = gu.torch()
    coords = synth.WORKLOADS["T"]()
    o = oracle.OracleGrid(coords)
    lib = vbm.load()
    import ctypes
    for log2w in (6, 8):
        g = vbm.vbm_build(coords, log2w)
        nb = g.info["n_blocks"]
        sides = [gu.to_dev(synth.sidecar_uniform(o.n, C, seed=C)) for C in CS]
        outs = [t.full_like(s, float("nan")) for s in sides]
        W = 1 << log2w
        cuts = [0, 1, nb // 3, nb - 1, nb]
        for b0, b1 in zip(cuts[:-1], cuts[1:]):
            sc = (ctypes.c_void_p * 4)(*[s.data_ptr() for s in sides])
            ou = (ctypes.c_void_p * 4)(*[x.data_ptr() for x in outs])
            cs = (ctypes.c_int * 4)(*CS)
            assert lib.vbm_box_filter_batch_blocks(g.handle, b0, b1, 4, sc, cs, ou, resolver, None) == 0
            t.cuda.synchronize()
            hi = min(o.n, b1 * W)
            for C, x in zip(CS, outs):  # rows past this range are still untouched
                assert np.isnan(x.cpu().numpy().reshape(-1, C)[hi + 1:]).all()
        for C, s, x in zip(CS, sides, outs):
            np.testing.assert_array_equal(gu.bits(x.cpu().numpy()), gu.bits(o.box_filter(s.cpu().numpy(), C)),
                                          err_msg=f"C={C} W={W}")
        sc = (ctypes.c_void_p * 1)(sides[0].data_ptr())
        ou = (ctypes.c_void_p * 1)(outs[1].data_ptr())
        cs = (ctypes.c_int * 1)(1)
        assert lib.vbm_box_filter_batch_blocks(g.handle, 2, 1, 1, sc, cs, ou, resolver, None) == -1
        assert lib.vbm_box_filter_batch_blocks(g.handle, 0, nb + 1, 1, sc, cs, ou, resolver, None) == -1


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _shard_rank(rank, world, port, workload, log2w, device_build, outdir):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import sparse_voxel_grid_gb300 as v
    import synth as syn
    from sparse_voxel_grid_gb300 import shard as sh
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        coords = syn.WORKLOADS[workload]()
        g = v.vbm_build_device(torch.from_numpy(coords).cuda(), log2w) if device_build else v.vbm_build(coords, log2w)
        plan = sh.ShardPlan(g, world, rank)
        lo, hi = plan.lo[rank], plan.hi[rank]
        sides, outs = [], []
        for C in CS:
            full = syn.sidecar_uniform(g.n, C, seed=0).reshape(-1, C)
            local = np.full_like(full, np.nan)  # rows this rank does not own stay NaN until the exchange
            local[lo:hi + 1] = full[lo:hi + 1]
            sides.append(torch.from_numpy(local.ravel()).cuda())
            outs.append(torch.full_like(sides[-1], float("nan")))
        sh.ShardedBoxFilter(g, plan).run(sides, CS, outs)
        torch.cuda.synchronize()
        for C, out in zip(CS, outs):
            rows = out.cpu().numpy().reshape(-1, C)
            np.save(os.path.join(outdir, f"r{rank}_C{C}.npy"), rows[lo:hi + 1])
            if rank == 0:
                np.save(os.path.join(outdir, f"row0_C{C}.npy"), rows[0])
    finally:
        dist.destroy_process_group()


def _run_shards(tmp_path, workload, log2w, world, device_build):
    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_shard_rank, args=(r, world, port, workload, log2w, device_build, str(tmp_path)))
             for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=600)
        assert p.exitcode == 0
    outs = []
    for C in CS:
        parts = [np.load(os.path.join(tmp_path, f"row0_C{C}.npy")).reshape(1, C)]
        parts += [np.load(os.path.join(tmp_path, f"r{r}_C{C}.npy")) for r in range(world)]
        outs.append(np.concatenate(parts).ravel())
    return outs


@pytest.mark.parametrize("log2w,world", [(6, 2), (7, 3)])
def test_sharded_filter_tiny_shell(tmp_path, log2w, world):
    coords = synth.WORKLOADS["T"]()
    o = oracle.OracleGrid(coords)
    got = _run_shards(tmp_path, "T", log2w, world, device_build=False)
    for C, x in zip(CS, got):
        want = o.box_filter(synth.sidecar_uniform(o.n, C, seed=0), C)
        np.testing.assert_array_equal(gu.bits(x), gu.bits(want), err_msg=f"C={C}")


def test_sharded_filter_shell_every_element(tmp_path):
    """The benchmarked workload (device-built S185 grid, W=512, C = 1, 3, 8, 16)
    in two shards: every output element against the oracle."""
    got = _run_shards(tmp_path, "S185", 9, 2, device_build=True)
    n = len(got[0]) - 1
    wants = oracle_pool.box_filter_all("S185", n, CS, seeds=(0, 0, 0, 0))
    for C, x, want in zip(CS, got, wants):
        np.testing.assert_array_equal(gu.bits(x), gu.bits(want), err_msg=f"C={C}")
