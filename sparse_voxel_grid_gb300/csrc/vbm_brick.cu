// Brick resolver: per-leaf padded neighbourhoods staged in shared memory.
//
// Sources (web pages; cited by title and section):
//   [2263] OpenVDB PR #2263 "Alternative stencil resolvers for VoxelBlockManager"
//   [2262] OpenVDB PR #2262 "NanoVDB VBM: Streaming box-stencil"
//
// The pages' cached resolver stages, per block, a table of neighbour-leaf
// pointers and then resolves every tap of every voxel with an in-leaf rank
// ([2263] "Summary").  On GB300 that costs ~50 instructions per tap and 27
// sidecar-row gathers per voxel through L1.  The brick resolver keeps the
// pages' structure (one CTA per VBM block, slots decoded in registers by the
// select-based decode, the same staged neighbour-leaf table, the same
// MaxCachedLeaves fallback to the tree walk) and adds one stage: for each leaf
// the block spans, the block builds a 10x10x10 brick covering the leaf and a
// one-voxel halo.  Cell (bx,by,bz) holds the leaf-relative position
// (bx-1, by-1, bz-1); its index is ranked once per z-row (one popcount for the
// row base, one per cell), and the brick holds the sidecar values of those
// indices (+0.0 for inactive cells).  Each voxel then reads its 27 taps at
// fixed offsets from its own cell and adds them in tap order
// t = (di+1)*9 + (dj+1)*3 + (dk+1) ([2262] "What changed").
//
// Bit-exactness: every tap's accumulator starts at +0.0 and adds in tap
// order.  An accumulator that starts at +0.0 is never -0.0 under
// round-to-nearest, and x + (+0.0) == x for every such x, so adding +0.0 for
// an inactive tap gives the same bits as skipping it.
//
// Only the brick planes that the block's voxels of that leaf touch are built
// (the leaf's voxels in the block cover a contiguous run of in-leaf offsets,
// hence a range of x planes).  Channels are processed in chunks of CCH: with
// one chunk the values are gathered while the row indices are in registers;
// with several, an index brick is built once and a value brick per chunk.
#include "vbm_launch.h"
#include "vbm_stencil.cuh"

namespace vbm {
namespace {

constexpr int kEdge = 10;        // brick edge: leaf-relative -1..8
constexpr int kCells = kEdge * kEdge * kEdge;

// The 10 indices of brick row (bx, by) of the leaf whose neighbour-table row is
// `trow` (27 leaf ids, (dx+1)*9 + (dy+1)*3 + (dz+1)).  Cell k holds
// leaf-relative z = k-1: cells 1..8 from the leaf at (dx,dy,0), cell 0 from
// (dx,dy,-1) (its z = 7) and cell 9 from (dx,dy,+1) (its z = 0).
__device__ __forceinline__ void brick_row(const LeafRec* __restrict__ leaves, const uint32_t* trow, int bx, int by,
                                          uint32_t (&idx)[kEdge]) {
    const int rx = bx - 1, ry = by - 1;                 // -1..8
    const int sx = (rx >> 3) + 1, sy = (ry >> 3) + 1;   // 0..2
    const uint32_t xw = (uint32_t)(rx & 7);             // mask word of plane x
    const uint32_t yb = (uint32_t)(ry & 7) * 8u;        // first bit of the z-row
    const uint32_t* col = trow + sx * 9 + sy * 3;
    uint32_t byte = 0, rb = 0;
    const uint32_t L = col[1];
    if (L != kNone) {
        const LeafRec* r = leaves + L;
        const uint64_t word = __ldg(&r->mask[xw]);
        byte = (uint32_t)(word >> yb) & 0xFFu;
        rb = __ldg(&r->base[xw]) + (uint32_t)__popcll(word & ((1ull << yb) - 1ull));
    }
#pragma unroll
    for (int z = 0; z < 8; ++z)
        idx[1 + z] = ((byte >> z) & 1u) ? rb + (uint32_t)__popc(byte & ((1u << z) - 1u)) : 0u;
    const uint32_t Lm = col[0], Lp = col[2];
    idx[0] = Lm != kNone ? leaf_index_at(leaves, Lm, xw * 64u + yb + 7u) : 0u;
    idx[kEdge - 1] = Lp != kNone ? leaf_index_at(leaves, Lp, xw * 64u + yb) : 0u;
}

// Sidecar chunk of one index into shared memory (zeros for index 0).
template <int CCH, bool VEC>
__device__ __forceinline__ void put_value(float* __restrict__ vb, int cell, const float* __restrict__ sc, uint32_t idx,
                                          int C, int ch0) {
    float v[CCH];
    if (idx) {
        load_row<CCH, VEC>(v, sc, idx, C, ch0);
    } else {
#pragma unroll
        for (int k = 0; k < CCH; ++k) v[k] = 0.0f;
    }
    if constexpr (CCH == 4) {
        reinterpret_cast<float4*>(vb)[cell] = make_float4(v[0], v[1], v[2], v[3]);
    } else if constexpr (CCH == 2) {
        reinterpret_cast<float2*>(vb)[cell] = make_float2(v[0], v[1]);
    } else {
#pragma unroll
        for (int k = 0; k < CCH; ++k) vb[cell * CCH + k] = v[k];
    }
}

template <int CCH>
__device__ __forceinline__ void get_value(float (&v)[CCH], const float* __restrict__ vb, int cell) {
    if constexpr (CCH == 4) {
        const float4 f = reinterpret_cast<const float4*>(vb)[cell];
        v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
    } else if constexpr (CCH == 2) {
        const float2 f = reinterpret_cast<const float2*>(vb)[cell];
        v[0] = f.x; v[1] = f.y;
    } else {
#pragma unroll
        for (int k = 0; k < CCH; ++k) v[k] = vb[cell * CCH + k];
    }
}

// Consumers reading a value brick; `cc` is the voxel's own cell.
template <int CCH>
__device__ __forceinline__ void brick_box(const float* __restrict__ vb, int cc, float (&acc)[CCH]) {
    float v[CCH];
#pragma unroll
    for (int k = 0; k < CCH; ++k) acc[k] = 0.0f;
#pragma unroll
    for (int t = 0; t < kBoxTaps; ++t) {
        get_value<CCH>(v, vb, cc + (t / 9 - 1) * 100 + ((t / 3) % 3 - 1) * 10 + (t % 3 - 1));
#pragma unroll
        for (int k = 0; k < CCH; ++k) acc[k] = __fadd_rn(acc[k], v[k]);
    }
}

template <int CCH, int OP>
__device__ __forceinline__ void brick_cross(const float* __restrict__ vb, int cc, float (&acc)[CCH]) {
    float v[CCH];
#pragma unroll
    for (int k = 0; k < CCH; ++k) acc[k] = 0.0f;
#pragma unroll
    for (int j = 0; j < kCrossTaps; ++j) {
        if (OP == VBM_CROSS_LAPLACIAN && j == 3) continue;
        get_value<CCH>(v, vb, cc + cross_di(j) * 100 + cross_dj(j) * 10 + cross_dk(j));
#pragma unroll
        for (int k = 0; k < CCH; ++k) acc[k] = __fadd_rn(acc[k], v[k]);
    }
    if constexpr (OP == VBM_CROSS_LAPLACIAN) {
        get_value<CCH>(v, vb, cc);
#pragma unroll
        for (int k = 0; k < CCH; ++k) acc[k] = __fsub_rn(acc[k], __fmul_rn(6.0f, v[k]));
    }
}

// Shared state of a block: staged table, per-slot offsets, leaf start slots.
struct BrickBlock {
    uint32_t b, W, fl, span, n_valid, index;
    const uint64_t* jb;
    bool active;
    Slot d;
};

// Decode the thread's slot; if the block fits the table, record its offset
// and leaf start, stage the neighbour-leaf table and synchronise.  Returns
// false (block-uniformly, before any barrier) when the block spans more than
// MaxCachedLeaves leaves.
__device__ __forceinline__ bool brick_prologue(const DevGrid& g, BrickBlock& k, uint32_t* table, uint16_t* offs,
                                               uint16_t* starts) {
    k.W = 1u << g.log2w;
    const uint32_t words = k.W >> 6;
    k.b = blockIdx.x;
    k.jb = g.jump + (size_t)k.b * words;
    k.fl = __ldg(&g.first_leaf[k.b]);
    k.span = block_span(k.jb, words);
    k.n_valid = min(k.W, g.n - k.b * k.W);
    const uint32_t s = threadIdx.x;
    k.active = s < k.n_valid;
    k.index = 1u + k.b * k.W + s;
    k.d.leaf = 0;
    k.d.off = 0;
    if (k.active) k.d = decode_slot(g, k.fl, k.jb, s, k.index);
    if (k.span > VBM_MAX_CACHED_LEAVES) return false;
    if (k.active) {
        offs[s] = (uint16_t)k.d.off;
        if (s == 0 || ((__ldg(&k.jb[s >> 6]) >> (s & 63u)) & 1ull)) starts[k.d.leaf - k.fl] = (uint16_t)s;
    }
    stage_leaf_table(g, k.fl, k.span, table);
    return true;
}

// Brick planes [x0, x1) that leaf l's voxels of this block need.
__device__ __forceinline__ void leaf_planes(const BrickBlock& k, const uint16_t* offs, const uint16_t* starts, uint32_t l,
                                            int& x0, int& x1) {
    const uint32_t sb = starts[l];
    const uint32_t se = (l + 1 < k.span) ? starts[l + 1] : k.n_valid;
    x0 = offs[sb] >> 6;
    x1 = (offs[se - 1] >> 6) + 3;
}

__device__ __forceinline__ int own_cell(const Slot& d) {
    return (int)(((d.off >> 6) + 1u) * 100u + (((d.off >> 3) & 7u) + 1u) * 10u + (d.off & 7u) + 1u);
}

// Fill the value brick planes [x0,x1) for channels [ch0, ch0+CCH).  From the
// index brick `ib` when given, else straight from the table row by rows.
template <int CCH, bool VEC>
__device__ __forceinline__ void fill_values(const DevGrid& g, const uint32_t* trow, const uint32_t* ib, float* vb,
                                            int x0, int x1, const float* __restrict__ sc, int C, int ch0) {
    if (ib) {
        for (int c = x0 * 100 + (int)threadIdx.x; c < x1 * 100; c += (int)blockDim.x)
            put_value<CCH, VEC>(vb, c, sc, ib[c], C, ch0);
    } else {
        for (int r = x0 * 10 + (int)threadIdx.x; r < x1 * 10; r += (int)blockDim.x) {
            uint32_t idx[kEdge];
            brick_row(g.leaves, trow, r / 10, r % 10, idx);
#pragma unroll
            for (int z = 0; z < kEdge; ++z) put_value<CCH, VEC>(vb, r * 10 + z, sc, idx[z], C, ch0);
        }
    }
}

__device__ __forceinline__ void fill_indices(const DevGrid& g, const uint32_t* trow, uint32_t* ib, int x0, int x1) {
    for (int r = x0 * 10 + (int)threadIdx.x; r < x1 * 10; r += (int)blockDim.x) {
        uint32_t idx[kEdge];
        brick_row(g.leaves, trow, r / 10, r % 10, idx);
#pragma unroll
        for (int z = 0; z < kEdge; ++z) ib[r * 10 + z] = idx[z];
    }
}

// KIND 0: 27-tap box; 1: cross Laplacian; 2: cross 7-tap sum.
template <int KIND, int CCH>
__device__ __forceinline__ void brick_consume(const float* vb, int cc, float (&acc)[CCH]) {
    if constexpr (KIND == 0) brick_box<CCH>(vb, cc, acc);
    else if constexpr (KIND == 1) brick_cross<CCH, VBM_CROSS_LAPLACIAN>(vb, cc, acc);
    else brick_cross<CCH, VBM_CROSS_SUM>(vb, cc, acc);
}

// Filter kernel.  Channels [ch_begin, ch_end) in chunks of CCH; MULTI: more
// than one chunk (index brick + value brick per chunk).
template <int KIND, int CCH, bool VEC, bool MULTI>
__global__ void __launch_bounds__(512) brick_filter_kernel(DevGrid g, const float* __restrict__ sc,
                                                           float* __restrict__ out, int C, int ch_begin, int ch_end) {
    __shared__ uint32_t table[VBM_MAX_CACHED_LEAVES * kBoxTaps];
    __shared__ uint16_t offs[512];
    __shared__ uint16_t starts[VBM_MAX_CACHED_LEAVES];
    __shared__ uint32_t ib[MULTI ? kCells : 1];
    __shared__ __align__(16) float vb[kCells * CCH];

    BrickBlock k;
    if (!brick_prologue(g, k, table, offs, starts)) {
        // MaxCachedLeaves fallback: per-tap tree walk, gathers from global memory.
        if (k.active) {
            for (int ch0 = ch_begin; ch0 < ch_end; ch0 += CCH) {
                if constexpr (KIND == 0) box_slot<CCH, VEC, false, false>(g, nullptr, k.d, k.index, sc, out, C, ch0);
                else if constexpr (KIND == 1)
                    cross_slot<CCH, VEC, false, VBM_CROSS_LAPLACIAN>(g, nullptr, k.d, k.index, sc, out, C, ch0);
                else cross_slot<CCH, VEC, false, VBM_CROSS_SUM>(g, nullptr, k.d, k.index, sc, out, C, ch0);
            }
        }
    } else {
        const uint32_t my_l = k.d.leaf - k.fl;
        const int cc = own_cell(k.d);
        for (uint32_t l = 0; l < k.span; ++l) {
            int x0, x1;
            leaf_planes(k, offs, starts, l, x0, x1);
            const uint32_t* trow = table + l * kBoxTaps;
            const bool mine = k.active && my_l == l;
            if constexpr (MULTI) {
                fill_indices(g, trow, ib, x0, x1);
                __syncthreads();
            }
            for (int ch0 = ch_begin; ch0 < ch_end; ch0 += CCH) {
                fill_values<CCH, VEC>(g, trow, MULTI ? ib : nullptr, vb, x0, x1, sc, C, ch0);
                __syncthreads();
                if (mine) {
                    float acc[CCH];
                    brick_consume<KIND, CCH>(vb, cc, acc);
                    store_row<CCH, VEC>(out, k.index, C, ch0, acc);
                }
                __syncthreads();
            }
        }
    }
    if (blockIdx.x == 0 && (int)threadIdx.x < ch_end - ch_begin) out[ch_begin + threadIdx.x] = 0.0f;
}

// Raw taps through the index brick.  SHAPE 27 (box) or 7 (cross).
template <int SHAPE>
__global__ void __launch_bounds__(512) brick_taps_kernel(DevGrid g, uint32_t* __restrict__ taps) {
    __shared__ uint32_t table[VBM_MAX_CACHED_LEAVES * kBoxTaps];
    __shared__ uint16_t offs[512];
    __shared__ uint16_t starts[VBM_MAX_CACHED_LEAVES];
    __shared__ uint32_t ib[kCells];

    BrickBlock k;
    if (!brick_prologue(g, k, table, offs, starts)) {
        if (k.active) {
            uint32_t* row = taps + (size_t)k.index * SHAPE;
            if constexpr (SHAPE == kBoxTaps) {
                const TapResolver<false> resolve(g, nullptr, k.d);
#pragma unroll
                for (int t = 0; t < kBoxTaps; ++t) row[t] = resolve(t / 9 - 1, (t / 3) % 3 - 1, t % 3 - 1);
            } else {
                uint32_t st[kCrossTaps];
                resolve_cross<false>(g, nullptr, k.d, st);
#pragma unroll
                for (int j = 0; j < kCrossTaps; ++j) row[j] = st[j];
            }
        }
    } else {
        const uint32_t my_l = k.d.leaf - k.fl;
        const int cc = own_cell(k.d);
        for (uint32_t l = 0; l < k.span; ++l) {
            int x0, x1;
            leaf_planes(k, offs, starts, l, x0, x1);
            fill_indices(g, table + l * kBoxTaps, ib, x0, x1);
            __syncthreads();
            if (k.active && my_l == l) {
                uint32_t* row = taps + (size_t)k.index * SHAPE;
                if constexpr (SHAPE == kBoxTaps) {
#pragma unroll
                    for (int t = 0; t < kBoxTaps; ++t)
                        row[t] = ib[cc + (t / 9 - 1) * 100 + ((t / 3) % 3 - 1) * 10 + (t % 3 - 1)];
                } else {
#pragma unroll
                    for (int j = 0; j < kCrossTaps; ++j) row[j] = ib[cc + cross_di(j) * 100 + cross_dj(j) * 10 + cross_dk(j)];
                }
            }
            __syncthreads();
        }
    }
    if (blockIdx.x == 0 && threadIdx.x < (unsigned)SHAPE) taps[threadIdx.x] = 0u;
}

template <int KIND, int CCH, bool VEC, bool MULTI>
cudaError_t launch_brick(const DevGrid& g, const float* sc, int C, int ch_begin, int ch_end, float* out,
                         cudaStream_t stream) {
    brick_filter_kernel<KIND, CCH, VEC, MULTI>
        <<<g.n_blocks, threads_for(g.log2w), 0, stream>>>(g, sc, out, C, ch_begin, ch_end);
    return cudaGetLastError();
}

template <int KIND>
cudaError_t launch_brick_kind(const DevGrid& g, const float* sc, int C, float* out, cudaStream_t stream) {
    switch (C) {
        case 1: return launch_brick<KIND, 1, false, false>(g, sc, C, 0, 1, out, stream);
        case 2: return launch_brick<KIND, 2, false, false>(g, sc, C, 0, 2, out, stream);
        case 3: return launch_brick<KIND, 3, false, false>(g, sc, C, 0, 3, out, stream);
        case 4: return launch_brick<KIND, 4, true, false>(g, sc, C, 0, 4, out, stream);
        default: break;
    }
    if (C % 4 == 0) return launch_brick<KIND, 4, true, true>(g, sc, C, 0, C, out, stream);
    // Rows are not 16-byte aligned: scalar loads; chunks of 4, then the rest.
    const int q = C / 4 * 4;
    cudaError_t e = q > 4 ? launch_brick<KIND, 4, false, true>(g, sc, C, 0, q, out, stream)
                          : launch_brick<KIND, 4, false, false>(g, sc, C, 0, 4, out, stream);
    if (e != cudaSuccess) return e;
    switch (C - q) {
        case 1: return launch_brick<KIND, 1, false, false>(g, sc, C, q, C, out, stream);
        case 2: return launch_brick<KIND, 2, false, false>(g, sc, C, q, C, out, stream);
        default: return launch_brick<KIND, 3, false, false>(g, sc, C, q, C, out, stream);
    }
}

}  // namespace

cudaError_t launch_brick_box(const DevGrid& g, const float* sidecar, int C, float* out, cudaStream_t stream) {
    return launch_brick_kind<0>(g, sidecar, C, out, stream);
}

cudaError_t launch_brick_cross(const DevGrid& g, const float* sidecar, int C, float* out, int op, cudaStream_t stream) {
    return op == VBM_CROSS_LAPLACIAN ? launch_brick_kind<1>(g, sidecar, C, out, stream)
                                     : launch_brick_kind<2>(g, sidecar, C, out, stream);
}

cudaError_t launch_brick_taps(const DevGrid& g, uint32_t* taps, int shape, cudaStream_t stream) {
    if (shape == kBoxTaps) brick_taps_kernel<kBoxTaps><<<g.n_blocks, threads_for(g.log2w), 0, stream>>>(g, taps);
    else brick_taps_kernel<kCrossTaps><<<g.n_blocks, threads_for(g.log2w), 0, stream>>>(g, taps);
    return cudaGetLastError();
}

}  // namespace vbm
