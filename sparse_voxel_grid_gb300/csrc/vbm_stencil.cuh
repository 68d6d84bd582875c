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

// acc[ch] += (idx != 0 ? sidecar[idx*C + ch0 + ch] : +0.0f) for ch < CC.  The
// load is predicated rather than branched around, so the loads of several taps
// can be in flight at once; an inactive tap adds +0.0, which leaves an fp32
// accumulator that started at +0.0 unchanged bit for bit (such a sum is never
// -0.0), so the result equals skipping the tap.
template <int CC, bool VEC>
__device__ __forceinline__ void gather_add_if(float (&acc)[CC], const float* __restrict__ sc, uint32_t idx, int C,
                                              int ch0) {
    const float* row = sc + (size_t)idx * (size_t)C + ch0;
    if constexpr (VEC) {
#pragma unroll
        for (int q = 0; q < CC / 4; ++q) {
            float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (idx) v = __ldg(reinterpret_cast<const float4*>(row) + q);
            acc[4 * q + 0] = __fadd_rn(acc[4 * q + 0], v.x);
            acc[4 * q + 1] = __fadd_rn(acc[4 * q + 1], v.y);
            acc[4 * q + 2] = __fadd_rn(acc[4 * q + 2], v.z);
            acc[4 * q + 3] = __fadd_rn(acc[4 * q + 3], v.w);
        }
    } else {
#pragma unroll
        for (int ch = 0; ch < CC; ++ch) {
            float v = 0.0f;
            if (idx) v = __ldg(row + ch);
            acc[ch] = __fadd_rn(acc[ch], v);
        }
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

template <int V>
struct IntC {
    static constexpr int value = V;
};

// f(IntC<0>{}) .. f(IntC<8>{}) in order, each with a compile-time value.
template <class F>
__device__ __forceinline__ void static_for_9(F&& f) {
    f(IntC<0>{}); f(IntC<1>{}); f(IntC<2>{}); f(IntC<3>{}); f(IntC<4>{});
    f(IntC<5>{}); f(IntC<6>{}); f(IntC<7>{}); f(IntC<8>{});
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
        if constexpr (TABLE) return cached_index(g->rowrank, row, x + di, y + dj, z + dk);
        else return walk_index(*g, x + di, y + dj, z + dk);
    }
};

// The three taps (di,dj,-1), (di,dj,0), (di,dj,+1) of a voxel at in-leaf
// position (x,y,z), through its leaf's staged table row.  The three positions
// lie in one z-row (x+di, y+dj) -- of one leaf, or past its z face at z = 0
// or 7 -- so that row's entry with its z halo (kRowRanks: its 8 mask bits, the
// index of its first bit and the indices of its two halo voxels) and one
// popcount of its bits below z rank all three (the z-1 bit, when set, is the
// last of those bits; the z+1 bit follows the centre).  Only where the row's
// leaf is absent can a face-crossing tap still be active, in the absent leaf's
// z neighbour: that rare case takes the table entry of the neighbour and its
// row rank.
template <int DI, int DJ>
__device__ __forceinline__ void cached_column(const DevGrid& g, const uint32_t* __restrict__ row, int32_t x, int32_t y,
                                              int32_t z, uint32_t (&idx)[3]) {
    const int32_t nx = x + DI, ny = y + DJ;
    const int32_t sxy = ((nx >> 3) + 1) * 9 + ((ny >> 3) + 1) * 3;
    const uint32_t r = (uint32_t)(nx & 7) * 8u + (uint32_t)(ny & 7), zu = (uint32_t)z;
    const bool lo = zu == 0u, hi = zu == 7u;
    const uint32_t L0 = row[sxy + 1];
    uint4 c = make_uint4(0u, 0u, 0u, 0u);
    if (L0 != kNone) {
        c = __ldg(&g.rowrank_z[(size_t)L0 * kRowRanks + r]);
    } else if (lo || hi) {
        const uint32_t Le = row[sxy + (lo ? 0 : 2)];
        if (Le != kNone) {
            const uint2 n = __ldg(&g.rowrank[(size_t)Le * kRowRanks + r]);
            // bit 7 of the -z neighbour's row (after its bits 0..6), or bit 0 of the +z neighbour's
            const uint32_t t = lo ? (((n.y >> 7) & 1u) ? n.x + (uint32_t)__popc(n.y & 0x7Fu) : 0u)
                                  : ((n.y & 1u) ? n.x : 0u);
            c.z = t; c.w = t;
        }
    }
    const uint32_t cnt = (uint32_t)__popc(c.y & ((1u << zu) - 1u));  // row bits below the centre
    const uint32_t b3 = ((c.y << 1) >> zu) & 7u;                    // bits z-1, z, z+1 (0 past the row's ends)
    const uint32_t bz = (b3 >> 1) & 1u;
    idx[1] = bz ? c.x + cnt : 0u;
    idx[0] = lo ? c.z : ((b3 & 1u) ? c.x + cnt - 1u : 0u);
    idx[2] = hi ? c.w : ((b3 & 4u) ? c.x + cnt + bz : 0u);
}

// The 27 box taps of one voxel in tap order, three at a time: column
// c = (di+1)*3 + (dj+1) holds taps 3c, 3c+1, 3c+2.
template <int C3>
__device__ __forceinline__ void box_column(const DevGrid& g, const uint32_t* table_row, int32_t x, int32_t y,
                                           int32_t z, uint32_t (&idx)[3]) {
    cached_column<C3 / 3 - 1, C3 % 3 - 1>(g, table_row, x, y, z, idx);
}

// 27-tap box filter of one voxel ([2262] "What changed"): taps in order
// t = (di+1)*9 + (dj+1)*3 + (dk+1); acc starts at +0.0; each non-zero tap adds
// its sidecar row.  MAT: the 27 indices are resolved into a per-thread array
// first (computeBoxStencil); otherwise each tap is consumed as it is resolved
// (forEachBoxStencil; the cached form resolves a column of three taps, then
// consumes them in order).  Same adds in the same order either way.
template <int CC, bool VEC, bool TABLE, bool MAT>
__device__ __forceinline__ void box_slot(const DevGrid& g, const uint32_t* table_row, const Slot& d, uint32_t index,
                                         const float* __restrict__ sc, float* __restrict__ out, int C, int ch0) {
    const TapResolver<TABLE> resolve(g, table_row, d);
    float acc[CC];
#pragma unroll
    for (int ch = 0; ch < CC; ++ch) acc[ch] = 0.0f;
    if constexpr (TABLE) {
        uint32_t st[MAT ? kBoxTaps : 3];
        auto column = [&](auto c3) {
            constexpr int c = decltype(c3)::value;
            uint32_t col[3];
            box_column<c>(g, table_row, resolve.x, resolve.y, resolve.z, col);
            if constexpr (MAT) {
                st[3 * c] = col[0]; st[3 * c + 1] = col[1]; st[3 * c + 2] = col[2];
            } else {
#pragma unroll
                for (int k = 0; k < 3; ++k) gather_add_if<CC, VEC>(acc, sc, col[k], C, ch0);
            }
        };
        static_for_9(column);
        if constexpr (MAT) {
#pragma unroll
            for (int t = 0; t < kBoxTaps; ++t) gather_add_if<CC, VEC>(acc, sc, st[t], C, ch0);
        }
    } else if constexpr (MAT) {
        uint32_t st[kBoxTaps];
#pragma unroll
        for (int t = 0; t < kBoxTaps; ++t) st[t] = resolve(t / 9 - 1, (t / 3) % 3 - 1, t % 3 - 1);
#pragma unroll
        for (int t = 0; t < kBoxTaps; ++t) gather_add_if<CC, VEC>(acc, sc, st[t], C, ch0);
    } else {
#pragma unroll
        for (int t = 0; t < kBoxTaps; ++t) {
            const uint32_t idx = resolve(t / 9 - 1, (t / 3) % 3 - 1, t % 3 - 1);
            gather_add_if<CC, VEC>(acc, sc, idx, C, ch0);
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

// Box tap t of cross tap j: (cross_di+1)*9 + (cross_dj+1)*3 + (cross_dk+1).
__device__ __forceinline__ constexpr int cross_box_tap(int j) {
    return (cross_di(j) + 1) * 9 + (cross_dj(j) + 1) * 3 + (cross_dk(j) + 1);
}

// Stage row[l*7 + j] = leaf holding tap j's position when it leaves leaf
// firstLeafID + l (entry 3: the leaf itself), for the block's spanned leaves
// (the pages' 16 x 7 cross table), copied from the face entries of the
// builder's neighbour rows.  Ends with a barrier.
__device__ __forceinline__ void stage_cross_table(const DevGrid& g, uint32_t first_leaf, uint32_t span,
                                                  uint32_t* __restrict__ table) {
    for (uint32_t e = threadIdx.x; e < span * (uint32_t)kCrossTaps; e += blockDim.x) {
        const uint32_t l = e / kCrossTaps, j = e - l * kCrossTaps;
        table[e] = __ldg(&g.nbr[(size_t)(first_leaf + l) * kNbrStride + cross_box_tap((int)j)]);
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
            st[j] = NL == kNone ? 0u : row_index_at(g.rowrank, NL, pack_off(nx, ny, nz));
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
        gather_add_if<CC, VEC>(acc, sc, st[j], C, ch0);
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
