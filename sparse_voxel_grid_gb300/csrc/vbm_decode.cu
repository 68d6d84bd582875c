// Select-based inverse-map decode kernel (OpenVDB PR #2258 "VBM select-based
// inverse-map decode", "What changed"): every output slot ranks itself into
// its leaf with a jumpMap popcount and finds its voxel by a select into the
// leaf mask through the 9-bit prefix directory.  O(1) per slot.  Output is
// structure-of-arrays: a 32-bit leaf index and a 16-bit voxel offset per slot,
// written coalesced.
//
// GB300 layout.  The work per slot is tiny; what bounds the kernel is the
// chain of dependent loads (block metadata -> leaf record -> mask word) and
// how many such chains are in flight.  So:
//   - one resident wave of CTAs, each owning an equal contiguous slot range
//     (no tail wave);
//   - the CTA stages the firstLeafID and jumpMap words of the blocks its range
//     overlaps in shared memory, with per-word popcount prefixes, so the rank
//     is a shared-memory lookup plus one popcount.  One staging (three
//     barriers) serves VBM_DECODE_STAGE chunks of 512 slots: with one per
//     chunk, warps waited at the barriers more than on any load (decode on
//     the 20.4M-slot grid D: 107 -> 96 us with eight chunks, 40 registers
//     and 12 CTAs per SM; at 16 CTAs the 32-register cap spills);
//   - each thread decodes a group of kGroup (8) consecutive slots a .. a+7,
//     a a multiple of 8, so the group lies in one block and one jumpMap word.
//     Slot a ranks and selects; slot a+i's leaf is a's plus the jumpMap bits
//     a+1 .. a+i, and its offset is the next set bit after slot a+i-1's (one
//     find-first-set in the same mask word, rarely a later word) or the first
//     set bit of the leaf that starts at a+i.  One rank and one select serve
//     eight slots, and the group is stored with 16-byte stores (decode on the
//     20.4M-slot grid D: 134 -> 107 us with pairs, whose second slot first
//     took its own rank; 96 -> 91 us when it took its leaf from the same
//     jumpMap word; 91 -> 74 us with groups of four, 67 us with eight);
//   - the loads of the group's leaf record and mask word come first, then the
//     select and the next-bit steps, so the chains of a warp's threads overlap;
//   - the word search reads the leaf's directory in its pre-added form, the
//     eight 32-bit per-word base indices (first index + set bits in the words
//     before), two 128-bit loads and seven 32-bit compares against the slot's
//     index, instead of unpacking seven 9-bit fields of a 64-bit word.  The
//     same comparisons, so the same word and rank; fewer instructions (decode
//     on D: 146 -> 134 us).
#include "vbm_device.cuh"
#include "vbm_launch.h"

namespace vbm {
namespace {

#ifndef VBM_DECODE_GROUP
#define VBM_DECODE_GROUP 8
#endif
#ifndef VBM_DECODE_GROUPS
#define VBM_DECODE_GROUPS 1
#endif
#ifndef VBM_DECODE_MIN_CTAS
#define VBM_DECODE_MIN_CTAS 12
#endif
#ifndef VBM_DECODE_STAGE
#define VBM_DECODE_STAGE 8
#endif
constexpr int kDecodeThreads = 128;
constexpr int kGroup = VBM_DECODE_GROUP;                    // consecutive slots per group (2, 4 or 8)
constexpr int kGroups = VBM_DECODE_GROUPS;                  // groups per thread per chunk
constexpr int kMaxRange = kDecodeThreads * kGroup * kGroups;  // slots per chunk
constexpr int kStageRange = 512 * VBM_DECODE_STAGE;         // slots per staging of block metadata
constexpr int kMaxBlocks = kStageRange / 64 + 2;            // blocks a staged range can overlap
constexpr int kMaxWords = 8;                                // jumpMap words per block (W = 512)
static_assert(kGroup == 2 || kGroup == 4 || kGroup == 8, "slot groups of 2, 4 or 8");
static_assert(kStageRange % kMaxRange == 0, "a staged range holds whole chunks");

// Position of the first set bit of leaf L's mask at word w or later (the leaf
// has one there); *cw / *cword receive that word's number and bits.
__device__ __forceinline__ uint32_t first_bit_from(const LeafRec* __restrict__ rec, uint32_t w, uint32_t* cw,
                                                   uint64_t* cword) {
    uint64_t m = 0;
    for (; w < 7u; ++w) {
        m = __ldg(&rec->mask[w]);
        if (m) break;
    }
    if (w == 7u) m = __ldg(&rec->mask[7]);
    *cw = w;
    *cword = m;
    return 64u * w + (uint32_t)__ffsll((long long)m) - 1u;
}

__global__ void __launch_bounds__(kDecodeThreads, VBM_DECODE_MIN_CTAS) decode_kernel(DevGrid g, uint32_t n_cta, uint32_t* __restrict__ leaf_index,
                                                                uint16_t* __restrict__ voxel_offset) {
    __shared__ uint32_t s_fl[kMaxBlocks];
    __shared__ uint64_t s_jw[kMaxBlocks][kMaxWords];
    __shared__ uint16_t s_cum[kMaxBlocks][kMaxWords];  // set bits in words 0..k-1 of the block's jumpMap

    const uint32_t log2w = (uint32_t)g.log2w, W = 1u << log2w, words = W >> 6;
    const uint64_t n_slots = (uint64_t)g.n_blocks << log2w;
    // The CTA's range [r0, r1), aligned to the slot groups.
    const uint32_t r0 = (uint32_t)(n_slots * blockIdx.x / n_cta) & ~(uint32_t)(kGroup - 1);
    const uint32_t r1 = (uint32_t)(n_slots * (blockIdx.x + 1) / n_cta) & ~(uint32_t)(kGroup - 1);
    for (uint32_t S0 = r0; S0 < r1; S0 += kStageRange) {  // uniform per CTA
        const uint32_t S1 = min(r1, S0 + (uint32_t)kStageRange);
        const uint32_t b0 = S0 >> log2w, nb = ((S1 - 1u) >> log2w) - b0 + 1u;

        // Block metadata of the staged range into shared memory.
        for (uint32_t e = threadIdx.x; e < nb * (words + 1u); e += blockDim.x) {
            const uint32_t bl = e / (words + 1u), k = e - bl * (words + 1u);
            if (k == 0) s_fl[bl] = __ldg(&g.first_leaf[b0 + bl]);
            else s_jw[bl][k - 1u] = __ldg(&g.jump[(size_t)(b0 + bl) * words + (k - 1u)]);
        }
        __syncthreads();
        if (threadIdx.x < nb) {
            uint32_t run = 0;
            for (uint32_t k = 0; k < words; ++k) {
                s_cum[threadIdx.x][k] = (uint16_t)run;
                run += (uint32_t)__popcll(s_jw[threadIdx.x][k]);
            }
        }
        __syncthreads();

        // Each thread decodes groups of kGroup consecutive slots a .. a+kGroup-1
        // (a a multiple of kGroup, so the group lies in one block and one
        // jumpMap word).  Slot a by rank + select; slot a+i's leaf is a's plus
        // the jumpMap bits a+1 .. a+i, and its offset the next set bit after
        // slot a+i-1's in the same leaf, or the first set bit of the leaf that
        // starts at a+i.
        for (uint32_t s0 = S0; s0 < S1; s0 += kMaxRange) {  // uniform per CTA; no barrier between chunks
        const uint32_t s1 = min(S1, s0 + (uint32_t)kMaxRange);
        uint32_t lf[kGroups][kGroup];
        uint4 blo[kGroups], bhi[kGroups];
#pragma unroll
        for (int k = 0; k < kGroups; ++k) {
            const uint32_t a = s0 + (uint32_t)kGroup * (threadIdx.x + (uint32_t)k * kDecodeThreads);
#pragma unroll
            for (int i = 0; i < kGroup; ++i) lf[k][i] = kNone;
            if (a < s1 && a < g.n) {  // index = a + 1 <= N
                const uint32_t bl = (a >> log2w) - b0, s = a & (W - 1u), ws = s >> 6;
                const uint64_t word = s_jw[bl][ws];
                const uint32_t sb = s & 63u;
                lf[k][0] = s_fl[bl] + s_cum[bl][ws] + (uint32_t)__popcll(word & ((2ull << sb) - 1ull));
#pragma unroll
                for (int i = 1; i < kGroup; ++i)
                    if (a + (uint32_t)i < g.n) lf[k][i] = lf[k][i - 1] + (uint32_t)((word >> (sb + (uint32_t)i)) & 1ull);
                const uint4* base = reinterpret_cast<const uint4*>(g.leaves[lf[k][0]].base);
                blo[k] = __ldg(base);
                bhi[k] = __ldg(base + 1);
            }
        }
        uint64_t word[kGroups];
        uint32_t wsel[kGroups], r[kGroups];
#pragma unroll
        for (int k = 0; k < kGroups; ++k) {
            if (lf[k][0] == kNone) continue;
            const uint32_t index = s0 + (uint32_t)kGroup * (threadIdx.x + (uint32_t)k * kDecodeThreads) + 1u;
            const uint32_t b[8] = {blo[k].x, blo[k].y, blo[k].z, blo[k].w, bhi[k].x, bhi[k].y, bhi[k].z, bhi[k].w};
            uint32_t w = 0, before = b[0];
#pragma unroll
            for (int f = 1; f < 8; ++f) {
                const bool at_or_below = b[f] <= index;
                w += at_or_below ? 1u : 0u;
                before = at_or_below ? b[f] : before;
            }
            wsel[k] = w;
            r[k] = index - before;
            word[k] = __ldg(&g.leaves[lf[k][0]].mask[w]);
        }
#pragma unroll
        for (int k = 0; k < kGroups; ++k) {
            const uint32_t a = s0 + (uint32_t)kGroup * (threadIdx.x + (uint32_t)k * kDecodeThreads);
            if (a >= s1) continue;
            uint32_t off[kGroup];
#pragma unroll
            for (int i = 0; i < kGroup; ++i) off[i] = kNoOffset;
            if (lf[k][0] != kNone) {
                uint32_t cw = wsel[k];      // mask word of the last decoded slot
                uint64_t cword = word[k];
                off[0] = 64u * cw + select64(cword, r[k]);
#pragma unroll
                for (int i = 1; i < kGroup; ++i) {
                    if (lf[k][i] == kNone) break;
                    if (lf[k][i] == lf[k][i - 1]) {  // the next set bit of the same leaf
                        const uint32_t bit = off[i - 1] & 63u;
                        const uint64_t rest = bit == 63u ? 0ull : cword & (~0ull << (bit + 1u));
                        off[i] = rest ? 64u * cw + (uint32_t)__ffsll((long long)rest) - 1u
                                      : first_bit_from(g.leaves + lf[k][i], cw + 1u, &cw, &cword);
                    } else {  // a leaf starts at slot a+i
                        off[i] = first_bit_from(g.leaves + lf[k][i], 0u, &cw, &cword);
                    }
                }
            }
            if constexpr (kGroup == 8) {
                uint4* li = reinterpret_cast<uint4*>(leaf_index) + (a >> 2);
                li[0] = make_uint4(lf[k][0], lf[k][1], lf[k][2], lf[k][3]);
                li[1] = make_uint4(lf[k][4], lf[k][5], lf[k][6], lf[k][7]);
                reinterpret_cast<uint4*>(voxel_offset)[a >> 3] =
                    make_uint4(off[0] | (off[1] << 16), off[2] | (off[3] << 16), off[4] | (off[5] << 16),
                               off[6] | (off[7] << 16));
            } else if constexpr (kGroup == 4) {
                reinterpret_cast<uint4*>(leaf_index)[a >> 2] = make_uint4(lf[k][0], lf[k][1], lf[k][2], lf[k][3]);
                reinterpret_cast<uint2*>(voxel_offset)[a >> 2] =
                    make_uint2(off[0] | (off[1] << 16), off[2] | (off[3] << 16));
            } else {
                reinterpret_cast<uint2*>(leaf_index)[a >> 1] = make_uint2(lf[k][0], lf[k][1]);
                reinterpret_cast<ushort2*>(voxel_offset)[a >> 1] = make_ushort2((uint16_t)off[0], (uint16_t)off[1]);
            }
        }
        }
        __syncthreads();  // the next staged range overwrites the metadata
    }
}

// Sweep decode: the design the select decode replaced (OpenVDB PR #2258,
// "What changed"), kept as its A/B baseline.  One CTA of W threads per block;
// the threads jointly sweep all 512 voxel slots of every leaf overlapping the
// block (the leaf holding the block's first index and the `popcount(jumpMap)`
// leaves that start inside it), compute each active voxel's index and keep the
// ones that fall inside the block: O(span x 512) work per block, with a
// data-dependent branch per voxel.  Output identical to the select decode.
__global__ void __launch_bounds__(512) sweep_decode_kernel(DevGrid g, uint32_t* __restrict__ leaf_index,
                                                           uint16_t* __restrict__ voxel_offset) {
    const uint32_t log2w = (uint32_t)g.log2w, W = 1u << log2w, words = W >> 6;
    const uint32_t b = blockIdx.x, tid = threadIdx.x;
    const uint32_t first = 1u + (b << log2w);  // index of the block's slot 0
    const uint32_t slot = (b << log2w) + tid;
    if (slot >= g.n) {  // index = slot + 1 > N
        leaf_index[slot] = kNone;
        voxel_offset[slot] = kNoOffset;
    }
    const uint32_t fl = __ldg(&g.first_leaf[b]);
    const uint32_t span = block_span(g.jump + (size_t)b * words, words);
    for (uint32_t l = 0; l < span; ++l) {
        for (uint32_t off = tid; off < 512u; off += W) {
            const uint32_t idx = leaf_index_at(g.leaves, fl + l, off);
            if (idx != 0 && idx - first < W) {
                leaf_index[idx - 1u] = fl + l;
                voxel_offset[idx - 1u] = (uint16_t)off;
            }
        }
    }
}

}  // namespace

cudaError_t launch_decode(const DevGrid& g, uint32_t* leaf_index, uint16_t* voxel_offset, cudaStream_t stream) {
    if (g.n_blocks == 0) return cudaSuccess;
    const uint64_t n_slots = (uint64_t)g.n_blocks << g.log2w;
    // One resident wave of CTAs, each with an equal share of the slots.
    // Resident CTAs per SM, queried once (thread-safe initialisation); a
    // failed query counts as one and its error is cleared, not reported.
    static const int per_sm = [] {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel, kDecodeThreads, 0) != cudaSuccess) {
            cudaGetLastError();
            n = 1;
        }
        return n < 1 ? 1 : n;
    }();
    uint64_t n_cta = (uint64_t)(g.sm_count > 0 ? g.sm_count : 1) * (uint64_t)per_sm;
    const uint64_t max_cta = (n_slots + 63) / 64;  // at least 64 slots per CTA
    if (n_cta > max_cta) n_cta = max_cta;
    decode_kernel<<<(unsigned)n_cta, kDecodeThreads, 0, stream>>>(g, (uint32_t)n_cta, leaf_index, voxel_offset);
    return cudaGetLastError();
}

cudaError_t launch_sweep_decode(const DevGrid& g, uint32_t* leaf_index, uint16_t* voxel_offset, cudaStream_t stream) {
    if (g.n_blocks == 0) return cudaSuccess;
    sweep_decode_kernel<<<(unsigned)g.n_blocks, threads_for(g.log2w), 0, stream>>>(g, leaf_index, voxel_offset);
    return cudaGetLastError();
}

}  // namespace vbm
