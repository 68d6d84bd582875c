// Per-voxel stencil consumers shared by the kernels: channel gathers, the
// tap resolvers of one decoded voxel (tree walk or cached table), and the
// 27-tap box / 7-tap cross consumers built on them.
//
// Sources (web pages; cited by title and section):
//   [2263] OpenVDB PR #2263 "Alternative stencil resolvers for VoxelBlockManager"
//   [2262] OpenVDB PR #2262 "NanoVDB VBM: Streaming box-stencil"
#pragma once

#include "vbm_device.cuh"

namespace vbm {

// acc[ch] += sidecar[idx*C + ch0 + ch] for ch < CC, fp32 round-to-nearest;
// VEC: the row is read as float4s (CC % 4 == 0, rows 16-byte aligned).
template <int CC, bool VEC>
__device__ __forceinline__ void gather_add(float (&acc)[CC], const float* __restrict__ sc, uint32_t idx, int C,
                                           int ch0) {
    const float* row = sc + (size_t)idx * (size_t)C + ch0;
    if constexpr (VEC) {
#pragma unroll
        for (int q = 0; q < CC / 4; ++q) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(row) + q);
            acc[4 * q + 0] = __fadd_rn(acc[4 * q + 0], v.x);
            acc[4 * q + 1] = __fadd_rn(acc[4 * q + 1], v.y);
            acc[4 * q + 2] = __fadd_rn(acc[4 * q + 2], v.z);
            acc[4 * q + 3] = __fadd_rn(acc[4 * q + 3], v.w);
        }
    } else {
#pragma unroll
        for (int ch = 0; ch < CC; ++ch) acc[ch] = __fadd_rn(acc[ch], __ldg(row + ch));
    }
}

template <int CC, bool VEC>
__device__ __forceinline__ void load_row(float (&v)[CC], const float* __restrict__ sc, uint32_t idx, int C, int ch0) {
    const float* row = sc + (size_t)idx * (size_t)C + ch0;
    if constexpr (VEC) {
#pragma unroll
        for (int q = 0; q < CC / 4; ++q) {
            const float4 f = __ldg(reinterpret_cast<const float4*>(row) + q);
            v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
        }
    } else {
#pragma unroll
        for (int ch = 0; ch < CC; ++ch) v[ch] = __ldg(row + ch);
    }
}

template <int CC, bool VEC>
__device__ __forceinline__ void store_row(float* __restrict__ out, uint32_t index, int C, int ch0,
                                          const float (&acc)[CC]) {
    float* row = out + (size_t)index * (size_t)C + ch0;
    if constexpr (VEC) {
#pragma unroll
        for (int q = 0; q < CC / 4; ++q)
            reinterpret_cast<float4*>(row)[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
    } else {
#pragma unroll
        for (int ch = 0; ch < CC; ++ch) row[ch] = acc[ch];
    }
}

// Resolves tap (di,dj,dk) of one decoded voxel.  TABLE: through the block's
// staged neighbour-leaf table row of the voxel's leaf; otherwise by tree walk.
template <bool TABLE>
struct TapResolver {
    const DevGrid* g;
    const uint32_t* row;  // TABLE: 27 neighbour-leaf ids of the voxel's leaf
    int32_t x, y, z;      // TABLE: in-leaf position (0..7); walk: absolute coordinate

    __device__ __forceinline__ TapResolver(const DevGrid& grid, const uint32_t* table_row, const Slot& d) : g(&grid) {
        const int32_t lx = (int32_t)(d.off >> 6), ly = (int32_t)((d.off >> 3) & 7u), lz = (int32_t)(d.off & 7u);
        if constexpr (TABLE) {
            row = table_row;
            x = lx; y = ly; z = lz;
        } else {
            row = nullptr;
            const LeafRec* r = grid.leaves + d.leaf;
            x = __ldg(&r->origin[0]) + lx;
            y = __ldg(&r->origin[1]) + ly;
            z = __ldg(&r->origin[2]) + lz;
        }
    }
    __device__ __forceinline__ uint32_t operator()(int di, int dj, int dk) const {
        if constexpr (TABLE) return cached_index(g->leaves, row, x + di, y + dj, z + dk);
        else return walk_index(*g, x + di, y + dj, z + dk);
    }
};

// 27-tap box filter of one voxel ([2262] "What changed"): taps in order
// t = (di+1)*9 + (dj+1)*3 + (dk+1); acc starts at +0.0; each non-zero tap adds
// its sidecar row.  MAT: the 27 indices are resolved into a per-thread array
// first (computeBoxStencil); otherwise each tap is consumed as it is resolved
// (forEachBoxStencil).  Same adds in the same order either way.
template <int CC, bool VEC, bool TABLE, bool MAT>
__device__ __forceinline__ void box_slot(const DevGrid& g, const uint32_t* table_row, const Slot& d, uint32_t index,
                                         const float* __restrict__ sc, float* __restrict__ out, int C, int ch0) {
    const TapResolver<TABLE> resolve(g, table_row, d);
    float acc[CC];
#pragma unroll
    for (int ch = 0; ch < CC; ++ch) acc[ch] = 0.0f;
    if constexpr (MAT) {
        uint32_t st[kBoxTaps];
#pragma unroll
        for (int t = 0; t < kBoxTaps; ++t) st[t] = resolve(t / 9 - 1, (t / 3) % 3 - 1, t % 3 - 1);
#pragma unroll
        for (int t = 0; t < kBoxTaps; ++t)
            if (st[t]) gather_add<CC, VEC>(acc, sc, st[t], C, ch0);
    } else {
#pragma unroll
        for (int t = 0; t < kBoxTaps; ++t) {
            const uint32_t idx = resolve(t / 9 - 1, (t / 3) % 3 - 1, t % 3 - 1);
            if (idx) gather_add<CC, VEC>(acc, sc, idx, C, ch0);
        }
    }
    store_row<CC, VEC>(out, index, C, ch0, acc);
}

// ---------------------------------------------------------------------------
// 7-tap cross: taps j = 0..6 are the box taps t = 4,10,12,13,14,16,22, i.e.
// offsets (-1,0,0), (0,-1,0), (0,0,-1), (0,0,0), (0,0,1), (0,1,0), (1,0,0).
// ---------------------------------------------------------------------------
__device__ __forceinline__ constexpr int cross_di(int j) { return j == 0 ? -1 : j == 6 ? 1 : 0; }
__device__ __forceinline__ constexpr int cross_dj(int j) { return j == 1 ? -1 : j == 5 ? 1 : 0; }
__device__ __forceinline__ constexpr int cross_dk(int j) { return j == 2 ? -1 : j == 4 ? 1 : 0; }

// Stage row[l*7 + j] = leaf holding tap j's position when it leaves leaf
// firstLeafID + l (entry 3: the leaf itself), for the block's spanned leaves
// (the pages' 16 x 7 cross table).  Ends with a barrier.
__device__ __forceinline__ void stage_cross_table(const DevGrid& g, uint32_t first_leaf, uint32_t span,
                                                  uint32_t* __restrict__ table) {
    for (uint32_t e = threadIdx.x; e < span * (uint32_t)kCrossTaps; e += blockDim.x) {
        const uint32_t l = e / kCrossTaps, j = e - l * kCrossTaps;
        const uint32_t L = first_leaf + l;
        uint32_t id = L;
        if (j != 3u) {
            const LeafRec* rec = g.leaves + L;
            id = find_leaf(g, __ldg(&rec->origin[0]) + 8 * cross_di((int)j), __ldg(&rec->origin[1]) + 8 * cross_dj((int)j),
                           __ldg(&rec->origin[2]) + 8 * cross_dk((int)j));
        }
        table[e] = id;
    }
    __syncthreads();
}

// Resolve the 7 cross taps of one decoded voxel into st[].
template <bool TABLE>
__device__ __forceinline__ void resolve_cross(const DevGrid& g, const uint32_t* table_row, const Slot& d,
                                              uint32_t (&st)[kCrossTaps]) {
    const int32_t lx = (int32_t)(d.off >> 6), ly = (int32_t)((d.off >> 3) & 7u), lz = (int32_t)(d.off & 7u);
    if constexpr (TABLE) {
#pragma unroll
        for (int j = 0; j < kCrossTaps; ++j) {
            const int32_t nx = lx + cross_di(j), ny = ly + cross_dj(j), nz = lz + cross_dk(j);
            const bool leaves_leaf = ((nx | ny | nz) & ~7) != 0;  // some coordinate is -1 or 8
            const uint32_t NL = table_row[leaves_leaf ? j : 3];
            st[j] = NL == kNone ? 0u : leaf_index_at(g.leaves, NL, pack_off(nx, ny, nz));
        }
    } else {
        const LeafRec* r = g.leaves + d.leaf;
        const int32_t x = __ldg(&r->origin[0]) + lx, y = __ldg(&r->origin[1]) + ly, z = __ldg(&r->origin[2]) + lz;
#pragma unroll
        for (int j = 0; j < kCrossTaps; ++j) st[j] = walk_index(g, x + cross_di(j), y + cross_dj(j), z + cross_dk(j));
    }
}

// Cross consumers on resolved taps.  Laplacian: s = +0.0 plus each active face
// value in increasing tap order, out = s - 6*centre with the product and the
// difference rounded separately.  Sum: the 7 taps in order.
template <int CC, bool VEC, int OP>
__device__ __forceinline__ void cross_consume(const uint32_t (&st)[kCrossTaps], uint32_t index,
                                              const float* __restrict__ sc, float* __restrict__ out, int C, int ch0) {
    float acc[CC], v[CC];
#pragma unroll
    for (int ch = 0; ch < CC; ++ch) acc[ch] = 0.0f;
#pragma unroll
    for (int j = 0; j < kCrossTaps; ++j) {
        if (OP == VBM_CROSS_LAPLACIAN && j == 3) continue;  // the centre enters below
        if (st[j]) {
            load_row<CC, VEC>(v, sc, st[j], C, ch0);
#pragma unroll
            for (int ch = 0; ch < CC; ++ch) acc[ch] = __fadd_rn(acc[ch], v[ch]);
        }
    }
    if constexpr (OP == VBM_CROSS_LAPLACIAN) {
        load_row<CC, VEC>(v, sc, index, C, ch0);
#pragma unroll
        for (int ch = 0; ch < CC; ++ch) acc[ch] = __fsub_rn(acc[ch], __fmul_rn(6.0f, v[ch]));
    }
    store_row<CC, VEC>(out, index, C, ch0, acc);
}

template <int CC, bool VEC, bool TABLE, int OP>
__device__ __forceinline__ void cross_slot(const DevGrid& g, const uint32_t* table_row, const Slot& d, uint32_t index,
                                           const float* __restrict__ sc, float* __restrict__ out, int C, int ch0) {
    uint32_t st[kCrossTaps];
    resolve_cross<TABLE>(g, table_row, d, st);
    cross_consume<CC, VEC, OP>(st, index, sc, out, C, ch0);
}

}  // namespace vbm
