// Brick resolver: per-leaf padded index bricks in shared memory, then a
// channel-parallel gather.
//
// Sources (web pages; cited by title and section):
//   [2263] OpenVDB PR #2263 "Alternative stencil resolvers for VoxelBlockManager"
//   [2262] OpenVDB PR #2262 "NanoVDB VBM: Streaming box-stencil"
//   [2258] OpenVDB PR #2258 "VBM select-based inverse-map decode"
//
// The pages' cached resolver stages, per VBM block, a table of neighbour-leaf
// pointers by probing the tree, then resolves every tap of every voxel with an
// in-leaf rank ([2263] "Summary").  Measured on GB300 that costs ~1,500
// instructions per voxel at one channel and, at 16 channels, 27 row gathers
// per voxel that saturate L1.  This resolver keeps the pages' structure (one CTA
// per VBM block; every slot decoded in registers by the select-based decode;
// a block's voxels span consecutive leaves firstLeafID .. firstLeafID +
// popcount(jumpMap)) and changes three things:
//
//  1. Neighbour-leaf ids come from the builder's per-leaf neighbour rows (27
//     ids in one 128-byte line) instead of 27 tree probes per spanned leaf.
//  2. For each spanned leaf the block builds a 10x10x10 brick of indices
//     covering the leaf and a one-voxel halo.  Cell (bx,by,bz) holds the index
//     of leaf-relative position (bx-1, by-1, bz-1), 0 if inactive.  A brick row
//     (fixed bx,by: ten z cells) costs one mask-word load, one popcount for the
//     row's base index and one popcount per cell (the in-leaf rank through the
//     per-word bases, i.e. the 9-bit directory pre-added to the leaf's first
//     index), plus one rank for each of the two halo cells.  Only the x planes
//     that the block's voxels of that leaf touch are built, and the rows of up
//     to max_group leaves are built together, one row per thread.
//  3. The gather is channel-parallel: thread (voxel, channel group) reads the
//     voxel's 27 tap indices from the brick at fixed offsets from its own cell,
//     in tap order t = (di+1)*9 + (dj+1)*3 + (dk+1), and adds
//     sidecar[idx*C + ch] for each non-zero tap ([2262] "What changed"), so the
//     lanes of one voxel read one contiguous sidecar row together.
//
// The adds per voxel and channel are the same as the other resolvers', in the
// same order, so the results are identical bit for bit.  There is no
// MaxCachedLeaves limit: blocks spanning more than max_group leaves are built
// in several rounds.
//
// Several sidecars on one grid (brick_box_shared_kernel): the decode and the
// index bricks do not depend on the sidecar, so one CTA per block builds them
// once and runs up to four sidecars' gathers from them; a C=1 and a C=3
// sidecar share one pass (each tap's index read once for both).
#include "vbm_brick.cuh"
#include "vbm_launch.h"
#include "vbm_stencil.cuh"

namespace vbm {
namespace {

using brick::BrickCtx;
using brick::brick_prologue;

constexpr int kEdge = 10;  // brick edge: leaf-relative -1..8
constexpr int kCells = kEdge * kEdge * kEdge;

// Leaves whose bricks are built in one round, by block width (shared memory
// max_group * 4000 bytes).  Measured per width on the shell: small blocks gain
// from the shared memory left to L1 and to more resident CTAs (W=64: 2 rather
// than 4 cut C=16 from 181 to 140 us; W=256: 4 rather than 6, 133 to 123 us);
// at W=512 one round for the ~5.5 spanned leaves matters more (8).
__host__ __device__ constexpr int max_group(int log2w) { return log2w <= 7 ? 2 : log2w == 8 ? 4 : 8; }

// Dynamic shared memory: ib[group][1000] index bricks, then offs[W] (voxel
// offset of each slot), lof[W] (slot's leaf - firstLeafID) and starts[span+1].
__host__ __device__ constexpr size_t brick_smem_bytes(int log2w) {
    return (size_t)max_group(log2w) * kCells * sizeof(uint32_t) + (size_t)3 * ((1u << log2w) + 1) * sizeof(uint16_t);
}

// The 10 indices of brick row (bx, by) of the leaf whose neighbour row is
// `nrow` (27 leaf ids at (dx+1)*9 + (dy+1)*3 + (dz+1)).  Cell k holds
// leaf-relative z = k-1: cells 1..8 from the leaf at (dx,dy,0), cell 0 from
// (dx,dy,-1) (its z = 7) and cell 9 from (dx,dy,+1) (its z = 0).  RR: ranked
// from the three leaves' row-rank entries of the z-row (kRowRanks); otherwise
// from their mask words and pre-added bases in the leaf records, which the
// decode has just read for the block's own leaves.
template <bool RR>
__device__ __forceinline__ void brick_row(const DevGrid& g, const uint32_t* __restrict__ nrow, int bx, int by,
                                          uint32_t (&idx)[kEdge]) {
    const int rx = bx - 1, ry = by - 1;                // -1..8
    const int sx = (rx >> 3) + 1, sy = (ry >> 3) + 1;  // 0..2
    const uint32_t* col = nrow + sx * 9 + sy * 3;
    const uint32_t Lm = __ldg(col), L0 = __ldg(col + 1), Lp = __ldg(col + 2);
    if constexpr (RR) {
        const uint32_t rr = (uint32_t)(rx & 7) * 8u + (uint32_t)(ry & 7);  // the z-row's entry
        uint2 c = make_uint2(0u, 0u), m = make_uint2(0u, 0u), p = make_uint2(0u, 0u);
        if (L0 != kNone) c = __ldg(&g.rowrank[(size_t)L0 * kRowRanks + rr]);
        if (Lm != kNone) m = __ldg(&g.rowrank[(size_t)Lm * kRowRanks + rr]);
        if (Lp != kNone) p = __ldg(&g.rowrank[(size_t)Lp * kRowRanks + rr]);
#pragma unroll
        for (int z = 0; z < 8; ++z)
            idx[1 + z] = ((c.y >> z) & 1u) ? c.x + (uint32_t)__popc(c.y & ((1u << z) - 1u)) : 0u;
        idx[0] = ((m.y >> 7) & 1u) ? m.x + (uint32_t)__popc(m.y & 0x7Fu) : 0u;  // z = 7 of the -z neighbour
        idx[kEdge - 1] = (p.y & 1u) ? p.x : 0u;                                // z = 0 of the +z neighbour
    } else {
        const uint32_t xw = (uint32_t)(rx & 7);       // mask word of plane x
        const uint32_t yb = (uint32_t)(ry & 7) * 8u;  // first bit of the z-row
        uint32_t byte = 0, rb = 0;
        if (L0 != kNone) {
            const LeafRec* r = g.leaves + L0;
            const uint64_t word = __ldg(&r->mask[xw]);
            byte = (uint32_t)(word >> yb) & 0xFFu;
            rb = __ldg(&r->base[xw]) + (uint32_t)__popcll(word & ((1ull << yb) - 1ull));
        }
#pragma unroll
        for (int z = 0; z < 8; ++z)
            idx[1 + z] = ((byte >> z) & 1u) ? rb + (uint32_t)__popc(byte & ((1u << z) - 1u)) : 0u;
        idx[0] = Lm != kNone ? leaf_index_at(g.leaves, Lm, xw * 64u + yb + 7u) : 0u;
        idx[kEdge - 1] = Lp != kNone ? leaf_index_at(g.leaves, Lp, xw * 64u + yb) : 0u;
    }
}

// Brick cell of a voxel's own position (its (0,0,0) tap).
__device__ __forceinline__ int own_cell(uint32_t off) {
    return (int)(((off >> 6) + 1u) * 100u + (((off >> 3) & 7u) + 1u) * 10u + (off & 7u) + 1u);
}

__device__ __forceinline__ constexpr int box_cell_delta(int t) { return (t / 9 - 1) * 100 + ((t / 3) % 3 - 1) * 10 + (t % 3 - 1); }
__device__ __forceinline__ constexpr int cross_cell_delta(int j) { return cross_di(j) * 100 + cross_dj(j) * 10 + cross_dk(j); }

// Build the bricks of spanned leaves l0 .. l0+nb-1 into ib[0..nb).  Leaf l's
// voxels in this block run from slot starts[l] to starts[l+1]-1, in increasing
// in-leaf offset (x-major), so they touch x planes x(first)-1 .. x(last)+1,
// i.e. brick planes [x(first), x(last)+3).  One row per thread.  VALUES (one
// channel only): store sidecar[idx] (+0.0 where idx == 0) instead of idx.
// Ends with a barrier.
template <bool VALUES, bool RR = VALUES>
__device__ __forceinline__ void build_round(const DevGrid& g, const BrickCtx& k, const uint16_t* offs,
                                            const uint16_t* starts, uint32_t l0, uint32_t nb, uint32_t* ib,
                                            const float* __restrict__ sc) {
    for (uint32_t r = threadIdx.x; r < nb * 100u; r += blockDim.x) {
        const uint32_t kk = r / 100u, row = r - kk * 100u, l = l0 + kk;
        const uint32_t x0 = offs[starts[l]] >> 6, x1 = (offs[starts[l + 1] - 1u] >> 6) + 3u;
        if (row < x0 * 10u || row >= x1 * 10u) continue;
        uint32_t idx[kEdge];
        brick_row<RR>(g, g.nbr + (size_t)(k.fl + l) * kNbrStride, (int)(row / 10u), (int)(row % 10u), idx);
        uint32_t* dst = ib + kk * kCells + row * kEdge;
        if constexpr (VALUES) {
            float v[kEdge];
#pragma unroll
            for (int z = 0; z < kEdge; ++z) v[z] = idx[z] ? __ldg(sc + idx[z]) : 0.0f;
#pragma unroll
            for (int z = 0; z < kEdge; ++z) dst[z] = __float_as_uint(v[z]);
        } else {
#pragma unroll
            for (int z = 0; z < kEdge; ++z) dst[z] = idx[z];
        }
    }
    __syncthreads();
}

// KIND 0: 27-tap box; 1: cross Laplacian; 2: cross 7-tap sum.  Channels
// [ch0, ch0+CC) of one voxel whose own brick cell is `cc` in brick `ibk`.
// acc[c] += sidecar[idx*C + ch0 + c] for c < CC, written without a branch: the
// load is predicated on idx != 0 and an inactive tap adds +0.0, which leaves
// an accumulator that started at +0.0 unchanged bit for bit.  CT > 0: the row
// stride C is the compile-time CT.
template <int CC, bool VEC, int CT>
__device__ __forceinline__ void gather_add_pred(float (&acc)[CC], const float* __restrict__ sc, uint32_t idx, int C,
                                                int ch0) {
    const uint32_t stride = CT > 0 ? (uint32_t)CT : (uint32_t)C;
    const float* row = sc + (size_t)idx * stride + ch0;
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
    } else if constexpr (CC == 3) {
        // A 12-byte row read as one 8-byte and one 4-byte load: the row's
        // float offset f has the parity of idx*stride + ch0, and the sidecar
        // is 16-byte aligned, so the 8-byte pair is (f, f+1) when f is even
        // and (f+1, f+2) when f is odd.  Two loads per tap instead of three.
        const bool odd = ((idx * stride + (uint32_t)ch0) & 1u) != 0u;
        float s = 0.0f;
        float2 p = make_float2(0.0f, 0.0f);
        if (idx) {
            s = __ldg(row + (odd ? 0 : 2));
            p = __ldg(reinterpret_cast<const float2*>(row + (odd ? 1 : 0)));
        }
        acc[0] = __fadd_rn(acc[0], odd ? s : p.x);
        acc[1] = __fadd_rn(acc[1], odd ? p.x : p.y);
        acc[2] = __fadd_rn(acc[2], odd ? p.y : s);
    } else {
#pragma unroll
        for (int c = 0; c < CC; ++c) {
            float v = 0.0f;
            if (idx) v = __ldg(row + c);
            acc[c] = __fadd_rn(acc[c], v);
        }
    }
}

// KIND 0: 27-tap box; 1: cross Laplacian; 2: cross 7-tap sum.  Channels
// [ch0, ch0+CC) of one voxel whose own brick cell is `cc` in brick `ibk`.
template <int KIND, int CC, bool VEC, int CT>
__device__ __forceinline__ void brick_consume(const uint32_t* __restrict__ ibk, int cc, uint32_t index,
                                              const float* __restrict__ sc, float* __restrict__ out, int C, int ch0) {
    const int Cs = CT > 0 ? CT : C;
    float acc[CC];
#pragma unroll
    for (int c = 0; c < CC; ++c) acc[c] = 0.0f;
    if constexpr (KIND == 0) {
#pragma unroll
        for (int t = 0; t < kBoxTaps; ++t) gather_add_pred<CC, VEC, CT>(acc, sc, ibk[cc + box_cell_delta(t)], Cs, ch0);
    } else {
#pragma unroll
        for (int j = 0; j < kCrossTaps; ++j) {
            if (KIND == 1 && j == 3) continue;  // the Laplacian's centre enters below
            gather_add_pred<CC, VEC, CT>(acc, sc, ibk[cc + cross_cell_delta(j)], Cs, ch0);
        }
        if constexpr (KIND == 1) {
            float v[CC];
            load_row<CC, VEC>(v, sc, index, Cs, ch0);
#pragma unroll
            for (int c = 0; c < CC; ++c) acc[c] = __fsub_rn(acc[c], __fmul_rn(6.0f, v[c]));
        }
    }
    store_row<CC, VEC>(out, index, Cs, ch0, acc);
}

// One-channel consumers reading a value brick (+0.0 in inactive cells; adding
// +0.0 to an fp32 sum that started at +0.0 leaves it unchanged bit for bit).
template <int KIND>
__device__ __forceinline__ float brick_consume_values(const uint32_t* __restrict__ vbk, int cc) {
    float acc = 0.0f;
    if constexpr (KIND == 0) {
#pragma unroll
        for (int t = 0; t < kBoxTaps; ++t) acc = __fadd_rn(acc, __uint_as_float(vbk[cc + box_cell_delta(t)]));
    } else {
#pragma unroll
        for (int j = 0; j < kCrossTaps; ++j) {
            if (KIND == 1 && j == 3) continue;
            acc = __fadd_rn(acc, __uint_as_float(vbk[cc + cross_cell_delta(j)]));
        }
        if constexpr (KIND == 1) acc = __fsub_rn(acc, __fmul_rn(6.0f, __uint_as_float(vbk[cc])));
    }
    return acc;
}

struct BrickSmem {
    uint32_t* ib;
    uint16_t *offs, *lof, *starts;
    uint32_t group;
};

__device__ __forceinline__ BrickSmem carve(unsigned char* smem, int log2w) {
    BrickSmem m;
    const uint32_t W1 = (1u << log2w) + 1u;
    m.group = (uint32_t)max_group(log2w);
    m.ib = reinterpret_cast<uint32_t*>(smem);
    m.offs = reinterpret_cast<uint16_t*>(m.ib + m.group * kCells);
    m.lof = m.offs + W1;
    m.starts = m.lof + W1;
    return m;
}

// The filter of VBM block b: channels [ch_begin, ch_begin + lanes*CC);
// `lanes` threads per voxel, each handling CC consecutive channels (VEC: as
// float4s).  VALUES: one channel, value bricks (lanes == CC == 1).
template <int KIND, int CC, bool VEC, bool VALUES, int CT>
__device__ __forceinline__ void brick_filter_block(const DevGrid& g, uint32_t b, const float* __restrict__ sc,
                                                   float* __restrict__ out, int C, int ch_begin, int lanes,
                                                   unsigned char* smem) {
    const BrickSmem m = carve(smem, g.log2w);
    BrickCtx k;
    brick_prologue<!VEC>(g, k, m.offs, m.lof, m.starts, b);
    const uint32_t L = CT > 0 ? (uint32_t)(CT / CC) : (uint32_t)lanes;
    for (uint32_t l0 = 0; l0 < k.span; l0 += m.group) {
        const uint32_t nb = min(m.group, k.span - l0);
        build_round<VALUES>(g, k, m.offs, m.starts, l0, nb, m.ib, sc);
        const uint32_t sb = m.starts[l0], se = m.starts[l0 + nb];
        if constexpr (VALUES) {
            for (uint32_t s = sb + threadIdx.x; s < se; s += blockDim.x) {
                const uint32_t* vbk = m.ib + (uint32_t)(m.lof[s] - l0) * kCells;
                out[1u + k.b * k.W + s] = brick_consume_values<KIND>(vbk, own_cell(m.offs[s]));
            }
        } else {
            const uint32_t items = (se - sb) * L;
            for (uint32_t it = threadIdx.x; it < items; it += blockDim.x) {
                const uint32_t v = L == 1 ? it : it / L, q = it - v * L, s = sb + v;
                const uint32_t* ibk = m.ib + (uint32_t)(m.lof[s] - l0) * kCells;
                brick_consume<KIND, CC, VEC, CT>(ibk, own_cell(m.offs[s]), 1u + k.b * k.W + s, sc, out, C,
                                             ch_begin + (int)(q * CC));
            }
        }
        __syncthreads();  // the next round overwrites the bricks
    }
    if (b == 0 && threadIdx.x < L * CC) out[ch_begin + threadIdx.x] = 0.0f;
}

template <int KIND, int CC, bool VEC, bool VALUES, int CT>
__global__ void __launch_bounds__(512) brick_filter_kernel(DevGrid g, const float* __restrict__ sc,
                                                           float* __restrict__ out, int C, int ch_begin, int lanes) {
    extern __shared__ __align__(16) unsigned char smem[];
    brick_filter_block<KIND, CC, VEC, VALUES, CT>(g, g.block0 + blockIdx.x, sc, out, C, ch_begin, lanes, smem);
}

// Several box filters of one grid in one launch.  The decode and the index
// bricks of a block do not depend on the sidecar, so one CTA per VBM block
// decodes the block and builds each round's bricks once, then runs the gather
// of every sidecar of the batch from them (channel counts with a compile-time
// layout only, see batch_width).  Measured on the shell for C = 1, 3, 8, 16:
// 220 us, against 312 us for four single-width launches and 262 us for one
// launch whose CTAs alternate between the sidecars.
constexpr int kMaxBatch = VBM_MAX_BATCH;  // include/vbm.h
constexpr int kFused = 4;                 // sidecars per launch
struct BoxBatch {
    const float* sc[kMaxBatch];
    float* out[kMaxBatch];
    int C[kMaxBatch];
    int count;
    int pair[2];  // entries (0,1) / (2,3) are gathered in one pass (pairs_in_one_pass)
};

__host__ __device__ constexpr bool batch_width(int C) {
    return C == 1 || C == 2 || C == 3 || C == 4 || C == 8 || C == 16;
}

// Two one-lane widths whose gathers share one pass (the host orders a pair
// by C).  C = 2 is left out: with its instances the kernel no longer fits
// its 40 registers without spills.
__host__ __device__ constexpr bool pairs_in_one_pass(int Ca, int Cb) {
    return (Ca == 1 || Ca == 3) && (Cb == 1 || Cb == 3) && Ca <= Cb;
}

// The gathers of one round for one sidecar, through the round's index bricks.
template <int CC, bool VEC, int CT>
__device__ __forceinline__ void round_gather(const BrickCtx& k, const BrickSmem& m, uint32_t l0, uint32_t sb,
                                             uint32_t se, uint32_t L, const float* __restrict__ sc,
                                             float* __restrict__ out, int C) {
    const uint32_t items = (se - sb) * L;
    for (uint32_t it = threadIdx.x; it < items; it += blockDim.x) {
        const uint32_t v = L == 1 ? it : it / L, q = it - v * L, s = sb + v;
        const uint32_t* ibk = m.ib + (uint32_t)(m.lof[s] - l0) * kCells;
        brick_consume<0, CC, VEC, CT>(ibk, own_cell(m.offs[s]), 1u + k.b * k.W + s, sc, out, C, (int)(q * CC));
    }
}

// The gather of sidecar E (< count) of the batch, its pointers passed as
// restrict-qualified kernel parameters so that the compiler may move the next
// voxel's loads above this voxel's stores (as in the single-width kernel;
// taken from a struct the pointers cost 10-15% of the gather's time).
template <int E>
__device__ __forceinline__ void gather_entry(const BrickCtx& k, const BrickSmem& m, uint32_t l0, uint32_t sb,
                                             uint32_t se, const BoxBatch& a, const float* __restrict__ sc,
                                             float* __restrict__ out) {
    if (E >= a.count) return;
    switch (a.C[E]) {  // uniform per CTA
        case 1: round_gather<1, false, 1>(k, m, l0, sb, se, 1, sc, out, 1); break;
        case 2: round_gather<2, false, 2>(k, m, l0, sb, se, 1, sc, out, 2); break;
        case 3: round_gather<3, false, 3>(k, m, l0, sb, se, 1, sc, out, 3); break;
        case 4: round_gather<4, true, 4>(k, m, l0, sb, se, 1, sc, out, 4); break;
        case 8: round_gather<4, true, 8>(k, m, l0, sb, se, 2, sc, out, 8); break;
        case 16: round_gather<4, true, 16>(k, m, l0, sb, se, 4, sc, out, 16); break;
        default: break;
    }
}

// The gathers of two one-lane sidecars (C = 1 or 3) in one pass over the
// round's voxels: each tap's index is read from the brick once for both, which
// saves the second pass's index reads (32 voxels per warp load, ~2.3
// wavefronts each from bank conflicts) and puts both rows' loads in flight
// together (the S185 four-sidecar step: 0.219 -> 0.210 ms).  Each sidecar's
// sums keep the tap order, so the results are those of two passes.
template <int CA, int CB>
__device__ __forceinline__ void round_gather_pair(const BrickCtx& k, const BrickSmem& m, uint32_t l0, uint32_t sb,
                                                  uint32_t se, const float* __restrict__ sa, float* __restrict__ oa,
                                                  const float* __restrict__ sbk, float* __restrict__ ob) {
    for (uint32_t s = sb + threadIdx.x; s < se; s += blockDim.x) {
        const uint32_t* ibk = m.ib + (uint32_t)(m.lof[s] - l0) * kCells;
        const int cc = own_cell(m.offs[s]);
        float acc_a[CA], acc_b[CB];
#pragma unroll
        for (int c = 0; c < CA; ++c) acc_a[c] = 0.0f;
#pragma unroll
        for (int c = 0; c < CB; ++c) acc_b[c] = 0.0f;
#pragma unroll
        for (int t = 0; t < kBoxTaps; ++t) {
            const uint32_t idx = ibk[cc + box_cell_delta(t)];
            gather_add_pred<CA, false, CA>(acc_a, sa, idx, CA, 0);
            gather_add_pred<CB, false, CB>(acc_b, sbk, idx, CB, 0);
        }
        const uint32_t index = 1u + k.b * k.W + s;
        store_row<CA, false>(oa, index, CA, 0, acc_a);
        store_row<CB, false>(ob, index, CB, 0, acc_b);
    }
}

template <int E>
__device__ __forceinline__ void gather_pair_entry(const BrickCtx& k, const BrickSmem& m, uint32_t l0, uint32_t sb,
                                                  uint32_t se, const BoxBatch& a, const float* __restrict__ sa,
                                                  float* __restrict__ oa, const float* __restrict__ sbk,
                                                  float* __restrict__ ob) {
    switch (a.C[E] * 4 + a.C[E + 1]) {  // uniform per CTA
        case 1 * 4 + 1: round_gather_pair<1, 1>(k, m, l0, sb, se, sa, oa, sbk, ob); break;
        case 1 * 4 + 3: round_gather_pair<1, 3>(k, m, l0, sb, se, sa, oa, sbk, ob); break;
        case 3 * 4 + 3: round_gather_pair<3, 3>(k, m, l0, sb, se, sa, oa, sbk, ob); break;
        default: break;
    }
}

// One CTA per VBM block for up to kFused sidecars: the block is decoded and
// each round's index bricks are built once, then every sidecar's gather runs
// from the same bricks.  40 registers (3 CTAs of 512 threads per SM): with
// the restrict-qualified pointers the extra registers hold more loads in
// flight (32 registers, 4 CTAs per SM, measured 8% slower).
__global__ void __launch_bounds__(512, 3) brick_box_shared_kernel(
    DevGrid g, BoxBatch a, const float* __restrict__ s0, const float* __restrict__ s1,
    const float* __restrict__ s2, const float* __restrict__ s3, float* __restrict__ o0, float* __restrict__ o1,
    float* __restrict__ o2, float* __restrict__ o3) {
    extern __shared__ __align__(16) unsigned char smem[];
    const BrickSmem m = carve(smem, g.log2w);
    BrickCtx k;
    brick_prologue<false>(g, k, m.offs, m.lof, m.starts, g.block0 + blockIdx.x);
    for (uint32_t l0 = 0; l0 < k.span; l0 += m.group) {
        const uint32_t nb = min(m.group, k.span - l0);
        build_round<false, true>(g, k, m.offs, m.starts, l0, nb, m.ib, nullptr);
        const uint32_t sb = m.starts[l0], se = m.starts[l0 + nb];
        if (a.pair[0]) {
            gather_pair_entry<0>(k, m, l0, sb, se, a, s0, o0, s1, o1);
        } else {
            gather_entry<0>(k, m, l0, sb, se, a, s0, o0);
            gather_entry<1>(k, m, l0, sb, se, a, s1, o1);
        }
        if (a.pair[1]) {
            gather_pair_entry<2>(k, m, l0, sb, se, a, s2, o2, s3, o3);
        } else {
            gather_entry<2>(k, m, l0, sb, se, a, s2, o2);
            gather_entry<3>(k, m, l0, sb, se, a, s3, o3);
        }
        __syncthreads();  // the next round overwrites the bricks
    }
    if (g.block0 + blockIdx.x == 0)
        for (int e = 0; e < a.count; ++e)
            for (uint32_t c = threadIdx.x; c < (uint32_t)a.C[e]; c += blockDim.x) a.out[e][c] = 0.0f;
}

// Raw taps through the index bricks.  SHAPE 27 (box) or 7 (cross).
template <int SHAPE>
__global__ void __launch_bounds__(512) brick_taps_kernel(DevGrid g, uint32_t* __restrict__ taps) {
    extern __shared__ __align__(16) unsigned char smem[];
    const BrickSmem m = carve(smem, g.log2w);
    BrickCtx k;
    brick_prologue<true>(g, k, m.offs, m.lof, m.starts, blockIdx.x);
    for (uint32_t l0 = 0; l0 < k.span; l0 += m.group) {
        const uint32_t nb = min(m.group, k.span - l0);
        build_round<false>(g, k, m.offs, m.starts, l0, nb, m.ib, nullptr);
        for (uint32_t s = m.starts[l0] + threadIdx.x; s < m.starts[l0 + nb]; s += blockDim.x) {
            const uint32_t* ibk = m.ib + (uint32_t)(m.lof[s] - l0) * kCells;
            const int cc = own_cell(m.offs[s]);
            uint32_t* row = taps + (size_t)(1u + k.b * k.W + s) * SHAPE;
            if constexpr (SHAPE == kBoxTaps) {
#pragma unroll
                for (int t = 0; t < kBoxTaps; ++t) row[t] = ibk[cc + box_cell_delta(t)];
            } else {
#pragma unroll
                for (int j = 0; j < kCrossTaps; ++j) row[j] = ibk[cc + cross_cell_delta(j)];
            }
        }
        __syncthreads();
    }
    if (blockIdx.x == 0 && threadIdx.x < (unsigned)SHAPE) taps[threadIdx.x] = 0u;
}

template <int KIND, int CC, bool VEC, bool VALUES, int CT = 0>
cudaError_t launch_brick(const DevGrid& g, const float* sc, int C, int lanes, float* out, cudaStream_t stream) {
    brick_filter_kernel<KIND, CC, VEC, VALUES, CT>
        <<<g.n_blocks, threads_for(g.log2w), brick_smem_bytes(g.log2w), stream>>>(g, sc, out, C, 0, lanes);
    return cudaGetLastError();
}

// Channel layout per C: one channel -> value bricks; 2 or 3 -> one lane with
// all channels; multiples of 4 -> lanes of kVecChannels channels read as
// float4s; anything else -> one lane per channel.
constexpr int kVecChannels = 4;

template <int KIND>
cudaError_t launch_brick_kind(const DevGrid& g, const float* sc, int C, float* out, cudaStream_t stream) {
    switch (C) {
        case 1: return launch_brick<KIND, 1, false, true, 1>(g, sc, C, 1, out, stream);
        case 2: return launch_brick<KIND, 2, false, false, 2>(g, sc, C, 1, out, stream);
        case 3: return launch_brick<KIND, 3, false, false, 3>(g, sc, C, 1, out, stream);
        case 4: return launch_brick<KIND, 4, true, false, 4>(g, sc, C, 1, out, stream);
        case 8: return launch_brick<KIND, 4, true, false, 8>(g, sc, C, 2, out, stream);
        case 16: return launch_brick<KIND, 4, true, false, 16>(g, sc, C, 4, out, stream);
        default: break;
    }
    if (C % kVecChannels == 0) return launch_brick<KIND, kVecChannels, true, false>(g, sc, C, C / kVecChannels, out, stream);
    if (C % 4 == 0) return launch_brick<KIND, 4, true, false>(g, sc, C, C / 4, out, stream);
    return launch_brick<KIND, 1, false, false>(g, sc, C, C, out, stream);
}

}  // namespace

size_t brick_box_smem_bytes(int log2w) { return brick_smem_bytes(log2w); }

cudaError_t launch_brick_box(const DevGrid& g, const float* sidecar, int C, float* out, cudaStream_t stream) {
    return launch_brick_kind<0>(g, sidecar, C, out, stream);
}

cudaError_t launch_brick_box_batch(const DevGrid& g, int count, const float* const* sidecars, const int* C,
                                   float* const* outs, cudaStream_t stream) {
    BoxBatch a{};
    a.count = 0;
    // Fused widths: C = 1, then C = 3 (so that they pair up), then the others.
    for (int pass = 0; pass < 3; ++pass)
        for (int i = 0; i < count; ++i) {
            const int rank = C[i] == 1 ? 0 : C[i] == 3 ? 1 : 2;
            if (!batch_width(C[i]) || rank != pass) continue;
            a.sc[a.count] = sidecars[i];
            a.out[a.count] = outs[i];
            a.C[a.count] = C[i];
            ++a.count;
        }
    for (int i = 0; i < count; ++i)
        if (!batch_width(C[i])) {
            const cudaError_t e = launch_brick_kind<0>(g, sidecars[i], C[i], outs[i], stream);
            if (e != cudaSuccess) return e;
        }
    // kFused sidecars per launch
    for (int first = 0; first < a.count; first += kFused) {
        BoxBatch part{};
        part.count = min(kFused, a.count - first);
        for (int i = 0; i < part.count; ++i) {
            part.sc[i] = a.sc[first + i];
            part.out[i] = a.out[first + i];
            part.C[i] = a.C[first + i];
        }
        for (int h = 0; h < 2; ++h)
            part.pair[h] = part.count >= 2 * h + 2 && pairs_in_one_pass(part.C[2 * h], part.C[2 * h + 1]);
        brick_box_shared_kernel<<<g.n_blocks, threads_for(g.log2w), brick_smem_bytes(g.log2w), stream>>>(
            g, part, part.sc[0], part.sc[1], part.sc[2], part.sc[3], part.out[0], part.out[1], part.out[2],
            part.out[3]);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_brick_cross(const DevGrid& g, const float* sidecar, int C, float* out, int op, cudaStream_t stream) {
    return op == VBM_CROSS_LAPLACIAN ? launch_brick_kind<1>(g, sidecar, C, out, stream)
                                     : launch_brick_kind<2>(g, sidecar, C, out, stream);
}

cudaError_t launch_brick_taps(const DevGrid& g, uint32_t* taps, int shape, cudaStream_t stream) {
    const size_t smem = brick_smem_bytes(g.log2w);
    const unsigned threads = (unsigned)threads_for(g.log2w);
    if (shape == kBoxTaps) brick_taps_kernel<kBoxTaps><<<g.n_blocks, threads, smem, stream>>>(g, taps);
    else brick_taps_kernel<kCrossTaps><<<g.n_blocks, threads, smem, stream>>>(g, taps);
    return cudaGetLastError();
}

}  // namespace vbm
