// Device functions shared by the VBM kernels: the select-based decode, the
// root-down tree walk, the in-leaf rank, and the cached neighbour-leaf table.
//
// Sources (web pages; cited by title and section):
//   [2263] OpenVDB PR #2263 "Alternative stencil resolvers for VoxelBlockManager"
//   [2258] OpenVDB PR #2258 "VBM select-based inverse-map decode"
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "vbm_internal.h"

namespace vbm {

// ---------------------------------------------------------------------------
// Bit primitives
// ---------------------------------------------------------------------------

// Position of the j-th (0-based) set bit of x; x must have more than j set
// bits.  Binary search over popcounts of halves (32, 16, 8, 4, 2, 1 bits).
__device__ __forceinline__ uint32_t select64(uint64_t x, uint32_t j) {
    uint32_t v = (uint32_t)x;
    uint32_t pos = 0;
    uint32_t c = __popc(v);
    if (j >= c) { j -= c; v = (uint32_t)(x >> 32); pos = 32; }
    c = __popc(v & 0xFFFFu);
    if (j >= c) { j -= c; v >>= 16; pos += 16; }
    c = __popc(v & 0xFFu);
    if (j >= c) { j -= c; v >>= 8; pos += 8; }
    c = __popc(v & 0xFu);
    if (j >= c) { j -= c; v >>= 4; pos += 4; }
    c = __popc(v & 0x3u);
    if (j >= c) { j -= c; v >>= 2; pos += 2; }
    c = v & 1u;
    if (j >= c) pos += 1;
    return pos;
}

// ---------------------------------------------------------------------------
// Decode ([2258] "What changed": rank into the block's jumpMap selects the
// leaf; select into the leaf's 512-bit mask, guided by the 9-bit prefix
// directory, recovers the voxel offset).  O(1) per slot, thread-local.
// ---------------------------------------------------------------------------

// Number of set jumpMap bits at or before slot s (bits 0..s of the block's
// W-bit map, words of 64).
__device__ __forceinline__ uint32_t jump_rank(const uint64_t* __restrict__ jb, uint32_t s) {
    const uint32_t ws = s >> 6;
    uint32_t r = 0;
    for (uint32_t k = 0; k < ws; ++k) r += __popcll(__ldg(&jb[k]));
    const uint64_t keep = (2ull << (s & 63)) - 1ull;  // bits 0..s&63 (all 64 when s&63 == 63)
    return r + __popcll(__ldg(&jb[ws]) & keep);
}

// Voxel offset of the r-th (0-based) active voxel of a leaf: the 9-bit
// directory (field w-1 = set bits in words 0..w-1) gives the word, an in-word
// select gives the bit.
__device__ __forceinline__ uint32_t leaf_select(const LeafRec* __restrict__ rec, uint32_t r) {
    const uint64_t P = __ldg(&rec->prefix);
    uint32_t w = 0;
#pragma unroll
    for (int f = 1; f < 8; ++f) w += (uint32_t)(((P >> (9 * (f - 1))) & 511u) <= r);
    const uint32_t before = w ? (uint32_t)((P >> (9 * (w - 1))) & 511u) : 0u;
    const uint64_t word = __ldg(&rec->mask[w]);
    return 64u * w + select64(word, r - before);
}

struct Slot {
    uint32_t leaf;
    uint32_t off;
};

// Decode slot s of block b (index = 1 + b*W + s <= N required).
__device__ __forceinline__ Slot decode_slot(const DevGrid& g, uint32_t first_leaf, const uint64_t* __restrict__ jb,
                                            uint32_t s, uint32_t index) {
    Slot out;
    out.leaf = first_leaf + jump_rank(jb, s);
    const LeafRec* rec = g.leaves + out.leaf;
    out.off = leaf_select(rec, index - __ldg(&rec->first));
    return out;
}

// ---------------------------------------------------------------------------
// Index of an in-leaf position: 0 if the bit is clear, else the leaf's base
// index for the word plus the set bits below it in that word.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t leaf_index_at(const LeafRec* __restrict__ leaves, uint32_t L, uint32_t off) {
    const LeafRec* r = leaves + L;
    const uint32_t w = off >> 6, bit = off & 63u;
    const uint64_t word = __ldg(&r->mask[w]);
    if (!((word >> bit) & 1ull)) return 0u;
    return __ldg(&r->base[w]) + (uint32_t)__popcll(word & ((1ull << bit) - 1ull));
}

// The same through the leaf's row ranks (kRowRanks): entry off>>3 is the z-row
// (x, y) of off = x*64 + y*8 + z; one 8-byte load and a popcount of the row's
// bits below z.
__device__ __forceinline__ uint32_t row_index_at(const uint2* __restrict__ rowrank, uint32_t L, uint32_t off) {
    const uint2 e = __ldg(&rowrank[(size_t)L * kRowRanks + (off >> 3)]);
    const uint32_t z = off & 7u;
    return ((e.y >> z) & 1u) ? e.x + (uint32_t)__popc(e.y & ((1u << z) - 1u)) : 0u;
}

__device__ __forceinline__ uint32_t pack_off(int32_t x, int32_t y, int32_t z) {
    return (uint32_t)((x & 7) << 6 | (y & 7) << 3 | (z & 7));
}

// ---------------------------------------------------------------------------
// Root-down tree walk ([2263] "Summary": each tap resolved by a root-down tree
// traversal; thread-local, no shared memory, safe from divergent threads).
// Root: binary search of the sorted upper-node keys; then the dense child
// tables of the upper (32^3) and lower (16^3) nodes.  Returns the leaf id or
// kNone.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t find_leaf(const DevGrid& g, int32_t x, int32_t y, int32_t z) {
    const uint64_t key = root_key_of(x, y, z);
    uint32_t lo = 0, hi = g.n_upper;
    while (lo < hi) {
        const uint32_t mid = (lo + hi) >> 1;
        if (__ldg(&g.root_keys[mid]) < key) lo = mid + 1; else hi = mid;
    }
    if (lo >= g.n_upper || __ldg(&g.root_keys[lo]) != key) return kNone;
    const uint32_t lower_slot = (uint32_t)(((x >> 7) & 31) << 10 | ((y >> 7) & 31) << 5 | ((z >> 7) & 31));
    const uint32_t lid = __ldg(&g.upper[(size_t)lo * kUpperSlots + lower_slot]);
    if (lid == kNone) return kNone;
    const uint32_t leaf_slot = (uint32_t)(((x >> 3) & 15) << 8 | ((y >> 3) & 15) << 4 | ((z >> 3) & 15));
    return __ldg(&g.lower[(size_t)lid * kLowerSlots + leaf_slot]);
}

// Index of the voxel at (x,y,z), 0 if inactive, by tree walk.
__device__ __forceinline__ uint32_t walk_index(const DevGrid& g, int32_t x, int32_t y, int32_t z) {
    const uint32_t L = find_leaf(g, x, y, z);
    return L == kNone ? 0u : row_index_at(g.rowrank, L, pack_off(x, y, z));
}

// ---------------------------------------------------------------------------
// Cached neighbour-leaf table ([2263] "Summary": the block cooperatively stages
// a per-leaf neighbour table in shared memory, built by all threads; "Built on
// the register-decode API": the staging derives what it needs from the block's
// metadata -- its first leaf is firstLeafID and it spans 1 + popcount(jumpMap)
// consecutive leaves).  Entry [l*27 + (dx+1)*9 + (dy+1)*3 + (dz+1)] is the id
// of the leaf whose origin is origin(firstLeafID+l) + 8*(dx,dy,dz), or kNone.
// The pages leave open how an entry is found; here it is copied from the
// builder's neighbour row of that leaf (the same 27 ids in one 128-byte line),
// so staging is one load per entry with no tree probe.  Must be called by
// every thread of the block; ends with a barrier.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void stage_leaf_table(const DevGrid& g, uint32_t first_leaf, uint32_t span,
                                                 uint32_t* __restrict__ table) {
    for (uint32_t e = threadIdx.x; e < span * 27u; e += blockDim.x) {
        const uint32_t l = e / 27u, t = e - l * 27u;
        table[e] = __ldg(&g.nbr[(size_t)(first_leaf + l) * kNbrStride + t]);
    }
    __syncthreads();
}

// Index of the in-leaf-relative position (nx,ny,nz), each in -1..8, of a voxel
// of table row `row` (the voxel's leaf is firstLeafID + row): which of the 27
// neighbour leaves holds it follows from floor(n/8), then an in-leaf rank.
__device__ __forceinline__ uint32_t cached_index(const uint2* __restrict__ rowrank, const uint32_t* __restrict__ row,
                                                 int32_t nx, int32_t ny, int32_t nz) {
    const int32_t slot = ((nx >> 3) + 1) * 9 + ((ny >> 3) + 1) * 3 + ((nz >> 3) + 1);
    const uint32_t NL = row[slot];
    return NL == kNone ? 0u : row_index_at(rowrank, NL, pack_off(nx, ny, nz));
}

// Number of leaves the block spans: 1 + popcount(jumpMap).
__device__ __forceinline__ uint32_t block_span(const uint64_t* __restrict__ jb, uint32_t words) {
    uint32_t span = 1;
    for (uint32_t k = 0; k < words; ++k) span += __popcll(__ldg(&jb[k]));
    return span;
}

}  // namespace vbm
