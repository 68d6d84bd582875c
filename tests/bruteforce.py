"""Brute force used to pin the CPU oracle on tiny grids.

Written independently of the oracle: the tree order is a depth-first walk of an
explicit nested node dictionary whose children are visited in lexicographic
order of their local (i, j, k) position (floor divisions, no bit packing), and
the stencils are Python-dictionary lookups of each neighbour coordinate, summed
tap by tap over whole numpy columns.  Only for grids of a few thousand voxels.
"""
from __future__ import annotations

import numpy as np

UPPER, LOWER, LEAF = 4096, 128, 8  # node edge lengths in voxels (32^3, 16^3, 8^3 children)


def tree_order(coords: np.ndarray) -> np.ndarray:
    """Coordinates in depth-first tree order: returns an (N,3) int64 array."""
    tree: dict = {}
    for x, y, z in np.asarray(coords, dtype=np.int64).tolist():
        u = (x // UPPER * UPPER, y // UPPER * UPPER, z // UPPER * UPPER)
        lo = ((x - u[0]) // LOWER, (y - u[1]) // LOWER, (z - u[2]) // LOWER)
        lo_org = (u[0] + lo[0] * LOWER, u[1] + lo[1] * LOWER, u[2] + lo[2] * LOWER)
        lf = ((x - lo_org[0]) // LEAF, (y - lo_org[1]) // LEAF, (z - lo_org[2]) // LEAF)
        lf_org = (lo_org[0] + lf[0] * LEAF, lo_org[1] + lf[1] * LEAF, lo_org[2] + lf[2] * LEAF)
        v = (x - lf_org[0], y - lf_org[1], z - lf_org[2])
        tree.setdefault(u, {}).setdefault(lo, {}).setdefault(lf, set()).add(v)
    out = []
    for u in sorted(tree):                      # root: upper origins, signed lexicographic
        for lo in sorted(tree[u]):              # lower nodes by local position in the upper node
            for lf in sorted(tree[u][lo]):      # leaves by local position in the lower node
                for v in sorted(tree[u][lo][lf]):  # voxels by local position in the leaf
                    out.append((u[0] + lo[0] * LOWER + lf[0] * LEAF + v[0],
                                u[1] + lo[1] * LOWER + lf[1] * LEAF + v[1],
                                u[2] + lo[2] * LOWER + lf[2] * LEAF + v[2]))
    return np.asarray(out, dtype=np.int64).reshape(-1, 3)


class Dense:
    """Brute-force stencil lookups over a grid given in index order.

    A Python dictionary maps each active coordinate to its index (position in
    the order + 1); any other point maps to 0."""

    def __init__(self, ordered: np.ndarray):
        self.ordered = np.asarray(ordered, dtype=np.int64)
        self.n = len(self.ordered)
        self.map = {tuple(p): i + 1 for i, p in enumerate(self.ordered.tolist())}
        self.lo = self.ordered.min(axis=0) - 1 if self.n else np.zeros(3, dtype=np.int64)
        hi = self.ordered.max(axis=0) + 1 if self.n else np.zeros(3, dtype=np.int64)
        self.shape = tuple((hi - self.lo + 1).tolist())

    def lookup(self, pts: np.ndarray) -> np.ndarray:
        m = self.map
        return np.array([m.get(tuple(p), 0) for p in np.asarray(pts, dtype=np.int64).tolist()], dtype=np.int64)

    def neighbour(self, di: int, dj: int, dk: int) -> np.ndarray:
        """Index of the (di,dj,dk) neighbour of each voxel, by index order."""
        m = self.map
        return np.array([m.get((x + di, y + dj, z + dk), 0) for x, y, z in self.ordered.tolist()], dtype=np.int64)

    def box_taps(self) -> np.ndarray:
        cols = [self.neighbour(di, dj, dk) for di in (-1, 0, 1) for dj in (-1, 0, 1) for dk in (-1, 0, 1)]
        return np.stack(cols, axis=1)

    FACES = ((-1, 0, 0), (0, -1, 0), (0, 0, -1), (0, 0, 1), (0, 1, 0), (1, 0, 0))

    def cross_taps(self) -> np.ndarray:
        order = [(-1, 0, 0), (0, -1, 0), (0, 0, -1), (0, 0, 0), (0, 0, 1), (0, 1, 0), (1, 0, 0)]
        return np.stack([self.neighbour(*d) for d in order], axis=1)

    @staticmethod
    def _values(sidecar: np.ndarray, C: int, nb: np.ndarray) -> np.ndarray:
        """Rows of the sidecar for neighbour indices; +0.0 where inactive.

        Adding +0.0 leaves any fp32 sum that started at +0.0 unchanged bit for
        bit (such a sum is never -0.0), so this equals skipping the tap."""
        rows = np.asarray(sidecar, dtype=np.float32).reshape(-1, C)[nb]
        rows[nb == 0] = np.float32(0.0)
        return rows

    def box_filter(self, sidecar: np.ndarray, C: int) -> np.ndarray:
        acc = np.zeros((self.n, C), dtype=np.float32)
        for di in (-1, 0, 1):
            for dj in (-1, 0, 1):
                for dk in (-1, 0, 1):
                    acc = acc + self._values(sidecar, C, self.neighbour(di, dj, dk))
        return acc

    def laplacian(self, sidecar: np.ndarray, C: int) -> np.ndarray:
        s = np.zeros((self.n, C), dtype=np.float32)
        for d in self.FACES:
            s = s + self._values(sidecar, C, self.neighbour(*d))
        centre = np.asarray(sidecar, dtype=np.float32).reshape(-1, C)[1:]
        return s - np.float32(6.0) * centre

