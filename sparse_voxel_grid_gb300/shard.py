"""Block-range shards of one grid over the ranks of a process group.

Every rank holds the whole grid (its topology is small: ~5 MB for the 1.29M-voxel
shell) and owns the sidecar rows of a contiguous range of VBM blocks
(vbm_shard_blocks).  To filter its blocks it needs, besides its own rows, its
halo: the rows of the neighbour leaves of its leaves that other ranks own
(vbm_shard_halo).  Since the topology is replicated, every rank computes every
rank's halo, so it knows which of its rows each other rank needs and no
request is exchanged: one all_to_all of packed rows per exchange.

The data path is the library's: vbm_gather_rows packs the rows to send,
vbm_scatter_rows places the received ones, vbm_box_filter_batch_blocks filters
the rank's blocks.  torch.distributed carries the packed rows (NCCL moves
device tensors; with gloo they pass through host memory).  The rank's sidecar
is a full (N+1)*C tensor in which only its own rows and its halo rows are
defined.
"""
from __future__ import annotations

import ctypes

import numpy as np

from ._lib import check, load


def shard_blocks(grid, n_shards: int) -> np.ndarray:
    """block_begin[0..n_shards]: shard s owns blocks block_begin[s] .. block_begin[s+1]-1."""
    out = np.empty(n_shards + 1, dtype=np.uint32)
    check(load().vbm_shard_blocks(grid.handle, int(n_shards), out.ctypes.data))
    return out


def shard_halo(grid, b0: int, b1: int) -> np.ndarray:
    """Sorted halo indices (uint32) of the shard owning blocks [b0, b1)."""
    lib = load()
    count = ctypes.c_uint64(0)
    check(lib.vbm_shard_halo(grid.handle, int(b0), int(b1), None, 0, ctypes.byref(count)))
    rows = np.empty(int(count.value), dtype=np.uint32)
    if rows.size:
        check(lib.vbm_shard_halo(grid.handle, int(b0), int(b1), rows.ctypes.data, rows.size, ctypes.byref(count)))
    return rows


class ShardPlan:
    """Who owns what, and which rows move where, for `world` shards of `grid`,
    seen from `rank`.  Host data only (numpy)."""

    def __init__(self, grid, world: int, rank: int):
        self.world, self.rank = int(world), int(rank)
        info = grid.info
        W, n = info["block_width"], info["n_active"]
        self.block_begin = shard_blocks(grid, world)
        b = self.block_begin.astype(np.int64)
        self.lo = [int(1 + b[q] * W) for q in range(world)]          # first owned index
        self.hi = [int(min(n, b[q + 1] * W)) for q in range(world)]  # last owned index
        self.halo = [shard_halo(grid, int(b[q]), int(b[q + 1])) for q in range(world)]
        r = self.rank
        mine = self.halo[r]
        # rows this rank sends to q: q's halo rows that this rank owns
        self.send_rows = [h[(h >= self.lo[r]) & (h <= self.hi[r])] for h in self.halo]
        # rows this rank receives from q: its halo rows that q owns (in halo order)
        self.recv_rows = [mine[(mine >= self.lo[q]) & (mine <= self.hi[q])] for q in range(world)]
        assert sum(len(x) for x in self.recv_rows) == len(mine)

    @property
    def blocks(self):
        return int(self.block_begin[self.rank]), int(self.block_begin[self.rank + 1])

    def send_order(self) -> np.ndarray:
        return np.concatenate(self.send_rows) if self.world else np.zeros(0, np.uint32)

    def recv_order(self) -> np.ndarray:
        return np.concatenate(self.recv_rows) if self.world else np.zeros(0, np.uint32)


def exchange_packed(plan: ShardPlan, sendbuf, C: int, group=None):
    """all_to_all of packed rows: sendbuf holds, for q = 0..world-1, the rows
    plan.send_rows[q] (C floats each); returns the received rows in the order
    of plan.recv_order().  Works on host tensors (gloo) and device tensors
    (NCCL)."""
    import torch
    import torch.distributed as dist
    in_splits = [len(x) * C for x in plan.send_rows]
    out_splits = [len(x) * C for x in plan.recv_rows]
    recv = torch.empty(sum(out_splits), dtype=sendbuf.dtype, device=sendbuf.device)
    dist.all_to_all_single(recv, sendbuf, out_splits, in_splits, group=group)
    return recv


class ShardedBoxFilter:
    """The box filter of this rank's blocks, with the halo exchanged first.

    `run(sidecars, Cs, outs, stream)`: sidecars are this rank's full-layout
    (N+1)*C CUDA tensors with its own rows filled; the call fills their halo
    rows from the other ranks, then writes this rank's output rows (and row 0
    on rank 0) of outs.  Collective: every rank of the group calls it with the
    same Cs.  `stream`: None (torch's current stream) or a torch.cuda.Stream;
    with gloo the exchange synchronises the device."""

    def __init__(self, grid, plan: ShardPlan, resolver=None, group=None):
        import torch
        import torch.distributed as dist
        from . import RESOLVE_BRICK
        self.grid, self.plan, self.group = grid, plan, group
        self.resolver = RESOLVE_BRICK if resolver is None else resolver
        self.via_host = dist.get_backend(group) != "nccl"
        self.send_idx = torch.from_numpy(plan.send_order().astype(np.int32)).cuda()
        self.recv_idx = torch.from_numpy(plan.recv_order().astype(np.int32)).cuda()

    def exchange(self, sidecar, C: int, stream=None) -> None:
        import torch
        from . import _stream_handle
        lib = load()
        s = _stream_handle(stream)
        sendbuf = torch.empty(len(self.send_idx) * C, dtype=torch.float32, device="cuda")
        ptr = ctypes.c_void_p(sidecar.data_ptr())
        if len(self.send_idx):
            check(lib.vbm_gather_rows(ptr, int(C), ctypes.c_void_p(self.send_idx.data_ptr()), len(self.send_idx),
                                      ctypes.c_void_p(sendbuf.data_ptr()), s))
        if self.via_host:  # gloo: the packed rows pass through host memory
            torch.cuda.synchronize()
            recv = exchange_packed(self.plan, sendbuf.cpu(), C, self.group).cuda()
            torch.cuda.synchronize()
        elif isinstance(stream, torch.cuda.Stream):
            # NCCL orders the collective after torch's current stream: make that
            # the stream the gather ran on, so the scatter below sees the rows
            with torch.cuda.stream(stream):
                recv = exchange_packed(self.plan, sendbuf, C, self.group)
        else:
            if stream is not None:
                raise TypeError("with NCCL, stream must be None or a torch.cuda.Stream")
            recv = exchange_packed(self.plan, sendbuf, C, self.group)
        if len(self.recv_idx):
            check(lib.vbm_scatter_rows(ctypes.c_void_p(recv.data_ptr()), int(C),
                                       ctypes.c_void_p(self.recv_idx.data_ptr()), len(self.recv_idx), ptr, s))

    def run(self, sidecars, Cs, outs, stream=None) -> None:
        import torch
        from . import _dev_ptr, _stream_handle
        for sd, C in zip(sidecars, Cs):
            self.exchange(sd, int(C), stream)
        k = len(sidecars)
        sc = (ctypes.c_void_p * k)()
        ou = (ctypes.c_void_p * k)()
        cs = (ctypes.c_int * k)()
        for i in range(k):
            m = (self.grid.n + 1) * int(Cs[i])
            sc[i] = _dev_ptr(sidecars[i], torch.float32, m, "sidecar").value
            ou[i] = _dev_ptr(outs[i], torch.float32, m, "out").value
            cs[i] = int(Cs[i])
        b0, b1 = self.plan.blocks
        check(load().vbm_box_filter_batch_blocks(self.grid.handle, b0, b1, k, sc, cs, ou, int(self.resolver),
                                                 _stream_handle(stream)))
