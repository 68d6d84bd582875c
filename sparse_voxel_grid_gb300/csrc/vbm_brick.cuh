// Per-block set-up shared by the brick kernels (vbm_brick.cu: box and cross;
// vbm_weno_brick.cu: WENO): one CTA per VBM block decodes every slot of its
// block into shared memory and records where each spanned leaf's slots start.
//
// Source (web page; cited by title and section):
//   [2258] OpenVDB PR #2258 "VBM select-based inverse-map decode"
#pragma once

#include "vbm_device.cuh"

namespace vbm {
namespace brick {

// Per-block state: block b of width W, its first leaf fl, the number of
// leaves it spans and of valid slots, its jumpMap words.  The prologues fill
// shared arrays offs[W] (voxel offset of each slot), lof[W] (slot's leaf -
// firstLeafID) and starts[span+1] (first slot of each spanned leaf;
// starts[span] = the valid slots).
struct BrickCtx {
    uint32_t b, W, fl, span, n_valid;
    const uint64_t* jb;
};

// Decode every valid slot of VBM block b (select-based decode, [2258] "What
// changed") into offs/lof and record where each spanned leaf starts.  Ends with
// a barrier.
__device__ __forceinline__ void brick_prologue_direct(const DevGrid& g, BrickCtx& k, uint16_t* offs, uint16_t* lof,
                                               uint16_t* starts, uint32_t b) {
    k.W = 1u << g.log2w;
    const uint32_t words = k.W >> 6;
    k.b = b;
    k.jb = g.jump + (size_t)k.b * words;
    k.fl = __ldg(&g.first_leaf[k.b]);
    k.span = block_span(k.jb, words);
    k.n_valid = min(k.W, g.n - k.b * k.W);
    for (uint32_t s = threadIdx.x; s < k.n_valid; s += blockDim.x) {
        const Slot d = decode_slot(g, k.fl, k.jb, s, 1u + k.b * k.W + s);
        offs[s] = (uint16_t)d.off;
        lof[s] = (uint16_t)(d.leaf - k.fl);
        if (s == 0 || ((__ldg(&k.jb[s >> 6]) >> (s & 63u)) & 1ull)) starts[d.leaf - k.fl] = (uint16_t)s;
    }
    if (threadIdx.x == 0) starts[k.span] = (uint16_t)k.n_valid;
    __syncthreads();
}

__device__ __forceinline__ void brick_prologue_staged(const DevGrid& g, BrickCtx& k, uint16_t* offs, uint16_t* lof,
                                               uint16_t* starts, uint32_t b) {
    // The block's jumpMap words and their popcount prefixes, staged once.
    __shared__ uint64_t s_jw[8];
    __shared__ uint32_t s_cum[9];
    k.W = 1u << g.log2w;
    const uint32_t words = k.W >> 6;
    k.b = b;
    k.jb = g.jump + (size_t)k.b * words;
    k.fl = __ldg(&g.first_leaf[k.b]);
    k.n_valid = min(k.W, g.n - k.b * k.W);
    if (threadIdx.x < 32u) {
        const uint32_t lane = threadIdx.x;
        const uint64_t w = lane < words ? __ldg(&k.jb[lane]) : 0ull;
        const uint32_t c = (uint32_t)__popcll(w);
        uint32_t incl = c;
#pragma unroll
        for (int d = 1; d < 8; d <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= (uint32_t)d) incl += t;
        }
        if (lane < words) {
            s_jw[lane] = w;
            s_cum[lane] = incl - c;
        }
        if (lane == words - 1u) s_cum[words] = incl;
    }
    __syncthreads();
    k.span = 1u + s_cum[words];
    for (uint32_t s = threadIdx.x; s < k.n_valid; s += blockDim.x) {
        const uint32_t ws = s >> 6;
        const uint64_t jw = s_jw[ws];
        const uint32_t leaf = k.fl + s_cum[ws] + (uint32_t)__popcll(jw & ((2ull << (s & 63u)) - 1ull));
        const LeafRec* rec = g.leaves + leaf;
        const uint32_t off = leaf_select(rec, 1u + k.b * k.W + s - __ldg(&rec->first));
        offs[s] = (uint16_t)off;
        lof[s] = (uint16_t)(leaf - k.fl);
        if (s == 0 || ((jw >> (s & 63u)) & 1ull)) starts[leaf - k.fl] = (uint16_t)s;
    }
    if (threadIdx.x == 0) starts[k.span] = (uint16_t)k.n_valid;
    __syncthreads();
}

// STAGED: jumpMap words and popcount prefixes in shared memory (faster for
// the one-lane layouts); otherwise each thread ranks from global memory
// (measured faster for the float4-lane layouts).
template <bool STAGED>
__device__ __forceinline__ void brick_prologue(const DevGrid& g, BrickCtx& k, uint16_t* offs, uint16_t* lof,
                                               uint16_t* starts, uint32_t b) {
    if constexpr (STAGED) brick_prologue_staged(g, k, offs, lof, starts, b);
    else brick_prologue_direct(g, k, offs, lof, starts, b);
}

}  // namespace brick
}  // namespace vbm
