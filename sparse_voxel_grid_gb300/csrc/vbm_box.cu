// 27-tap box stencil: fused decode + resolve + gather/accumulate filter, and
// the raw-tap export used for byte-exact validation.
//
// Sources (web pages; cited by title and section):
//   [2263] OpenVDB PR #2263 "Alternative stencil resolvers for VoxelBlockManager"
//   [2262] OpenVDB PR #2262 "NanoVDB VBM: Streaming box-stencil"
//
// One CTA per VBM block, one thread per slot.  Each thread decodes its slot in
// registers, resolves the 27 taps in order t = (di+1)*9 + (dj+1)*3 + (dk+1)
// ([2262] "What changed") either by tree walk or through the block's cached
// neighbour-leaf table ([2263] "Summary"), and for each non-zero tap adds
// sidecar[idx*C + ch] to a per-channel fp32 accumulator that starts at +0.0.
// Streamed: each tap is consumed as soon as it is resolved (forEachBoxStencil);
// materialised: all 27 indices are resolved into a per-thread array first
// (computeBoxStencil).  Both add the same values in the same order, so the
// results are identical bit for bit ([2262] "Validation").
#include "vbm_launch.h"
#include "vbm_stencil.cuh"

namespace vbm {
namespace {

// One CTA per VBM block, one thread per slot.  CT > 0: the row stride C is the
// compile-time CT (and ch0 is 0), so that the gathers' row addresses need no
// multiply by a runtime channel count.
template <int CC, bool VEC, bool CACHED, bool MAT, int CT>
__device__ __forceinline__ void box_filter_block(const DevGrid& g, const float* __restrict__ sc,
                                                 float* __restrict__ out, int C_rt, int ch0_rt) {
    const int C = CT > 0 ? CT : C_rt, ch0 = CT > 0 ? 0 : ch0_rt;
    __shared__ uint32_t table[CACHED ? VBM_MAX_CACHED_LEAVES * kBoxTaps : 1];
    const uint32_t W = 1u << g.log2w, words = W >> 6;
    const uint32_t b = g.block0 + blockIdx.x;
    const uint64_t* jb = g.jump + (size_t)b * words;
    const uint32_t fl = __ldg(&g.first_leaf[b]);
    // One slot per thread (blockDim == W).  The slot is decoded before the
    // cached table is staged: the decode's loads do not depend on the table,
    // so they are in flight while the staging's are.
    const uint32_t s = threadIdx.x, index = 1u + b * W + s;
    const bool valid = s < W && index <= g.n;
    Slot d{0u, 0u};
    if (valid) d = decode_slot(g, fl, jb, s, index);
    bool use_table = false;
    if constexpr (CACHED) {
        const uint32_t span = block_span(jb, words);
        use_table = span <= VBM_MAX_CACHED_LEAVES;  // block-uniform: the barrier inside is safe
        if (use_table) stage_leaf_table(g, fl, span, table);
    }
    if (valid) {
        if (CACHED && use_table) box_slot<CC, VEC, true, MAT>(g, table + (d.leaf - fl) * kBoxTaps, d, index, sc, out, C, ch0);
        else box_slot<CC, VEC, false, MAT>(g, nullptr, d, index, sc, out, C, ch0);
    }
    if (b == 0 && threadIdx.x < (unsigned)CC) out[ch0 + threadIdx.x] = 0.0f;
}

// The streamed one-lane forms (CC <= 3) run under a register bound: the cached
// ones at 32 (4 CTAs of 512 threads, 16 of 128, per SM; 48.7-49.2 against
// 51.2 us at 40 for C=1 on the 1.29M-voxel shell at W=128), the tree-walk ones
// at 40 (they spill at 32).  Left free, the cached C=1 kernel took 54 and ran
// 7-15% slower with fewer CTAs resident.  The wider and materialised forms
// would spill under these caps and keep the compiler's choice.
template <int CC, bool VEC, bool CACHED, bool MAT, int CT>
__global__ void __launch_bounds__(512) box_filter_kernel(DevGrid g, const float* __restrict__ sc,
                                                         float* __restrict__ out, int C, int ch0) {
    box_filter_block<CC, VEC, CACHED, MAT, CT>(g, sc, out, C, ch0);
}

template <int CC, bool VEC, bool CACHED, bool MAT, int CT>
__global__ void __launch_bounds__(512, 3) box_filter_kernel_r40(DevGrid g, const float* __restrict__ sc,
                                                                float* __restrict__ out, int C, int ch0) {
    box_filter_block<CC, VEC, CACHED, MAT, CT>(g, sc, out, C, ch0);
}

template <int CC, bool VEC, bool CACHED, bool MAT, int CT>
__global__ void __launch_bounds__(512, 4) box_filter_kernel_r32(DevGrid g, const float* __restrict__ sc,
                                                                float* __restrict__ out, int C, int ch0) {
    box_filter_block<CC, VEC, CACHED, MAT, CT>(g, sc, out, C, ch0);
}

// The materialised forms are held to 64 registers (2 CTAs of 512 threads per
// SM): with a compile-time stride the C=16 ones otherwise take 78-82 and run
// 11-28% slower.
template <int CC, bool VEC, bool CACHED, bool MAT, int CT>
__global__ void __launch_bounds__(512, 2) box_filter_kernel_r64(DevGrid g, const float* __restrict__ sc,
                                                                float* __restrict__ out, int C, int ch0) {
    box_filter_block<CC, VEC, CACHED, MAT, CT>(g, sc, out, C, ch0);
}

template <int CC, bool VEC, bool CACHED, bool MAT, int CT>
void launch_box_kernel(dim3 grid, dim3 block, cudaStream_t stream, const DevGrid& g, const float* sc, float* out,
                       int C, int ch0) {
    if constexpr (MAT) box_filter_kernel_r64<CC, VEC, CACHED, MAT, CT><<<grid, block, 0, stream>>>(g, sc, out, C, ch0);
    else if constexpr (CC <= 3 && CACHED) box_filter_kernel_r32<CC, VEC, CACHED, MAT, CT><<<grid, block, 0, stream>>>(g, sc, out, C, ch0);
    else if constexpr (CC <= 3) box_filter_kernel_r40<CC, VEC, CACHED, MAT, CT><<<grid, block, 0, stream>>>(g, sc, out, C, ch0);
    else box_filter_kernel<CC, VEC, CACHED, MAT, CT><<<grid, block, 0, stream>>>(g, sc, out, C, ch0);
}

// Raw taps: taps[index*27 + t].  Row 0 is zero.
template <bool CACHED>
__global__ void __launch_bounds__(512) box_taps_kernel(DevGrid g, uint32_t* __restrict__ taps) {
    __shared__ uint32_t table[CACHED ? VBM_MAX_CACHED_LEAVES * kBoxTaps : 1];
    const uint32_t W = 1u << g.log2w, words = W >> 6;
    const uint32_t b = blockIdx.x;
    const uint64_t* jb = g.jump + (size_t)b * words;
    const uint32_t fl = __ldg(&g.first_leaf[b]);
    bool use_table = false;
    if constexpr (CACHED) {
        const uint32_t span = block_span(jb, words);
        use_table = span <= VBM_MAX_CACHED_LEAVES;
        if (use_table) stage_leaf_table(g, fl, span, table);
    }
    for (uint32_t s = threadIdx.x; s < W; s += blockDim.x) {
        const uint32_t index = 1u + b * W + s;
        if (index > g.n) break;
        const Slot d = decode_slot(g, fl, jb, s, index);
        uint32_t* row = taps + (size_t)index * kBoxTaps;
        if (CACHED && use_table) {
            const TapResolver<true> resolve(g, table + (d.leaf - fl) * kBoxTaps, d);
#pragma unroll
            for (int t = 0; t < kBoxTaps; ++t) row[t] = resolve(t / 9 - 1, (t / 3) % 3 - 1, t % 3 - 1);
        } else {
            const TapResolver<false> resolve(g, nullptr, d);
#pragma unroll
            for (int t = 0; t < kBoxTaps; ++t) row[t] = resolve(t / 9 - 1, (t / 3) % 3 - 1, t % 3 - 1);
        }
    }
    if (b == 0 && threadIdx.x < (unsigned)kBoxTaps) taps[threadIdx.x] = 0u;
}

template <int CC, bool VEC, int CT = 0>
cudaError_t launch_box_cc(const DevGrid& g, const float* sc, int C, int ch0, float* out, int resolver, int output,
                          cudaStream_t stream) {
    const dim3 grid(g.n_blocks), block(threads_for(g.log2w));
    const bool cached = resolver == VBM_RESOLVE_CACHED, mat = output == VBM_OUTPUT_MATERIALISED;
    if (cached && mat) launch_box_kernel<CC, VEC, true, true, CT>(grid, block, stream, g, sc, out, C, ch0);
    else if (cached) launch_box_kernel<CC, VEC, true, false, CT>(grid, block, stream, g, sc, out, C, ch0);
    else if (mat) launch_box_kernel<CC, VEC, false, true, CT>(grid, block, stream, g, sc, out, C, ch0);
    else launch_box_kernel<CC, VEC, false, false, CT>(grid, block, stream, g, sc, out, C, ch0);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_box_filter(const DevGrid& g, const float* sidecar, int C, float* out, int resolver, int output,
                              cudaStream_t stream) {
    if (g.n_blocks == 0) {
        // Empty grid: only row 0 exists.
        return cudaMemsetAsync(out, 0, sizeof(float) * (size_t)C, stream);
    }
    switch (C) {
        case 1: return launch_box_cc<1, false, 1>(g, sidecar, C, 0, out, resolver, output, stream);
        case 2: return launch_box_cc<2, false, 2>(g, sidecar, C, 0, out, resolver, output, stream);
        case 3: return launch_box_cc<3, false, 3>(g, sidecar, C, 0, out, resolver, output, stream);
        case 4: return launch_box_cc<4, true, 4>(g, sidecar, C, 0, out, resolver, output, stream);
        case 8: return launch_box_cc<8, true, 8>(g, sidecar, C, 0, out, resolver, output, stream);
        case 16: return launch_box_cc<16, true, 16>(g, sidecar, C, 0, out, resolver, output, stream);
        default: break;
    }
    // Other widths: chunks of 4 channels (scalar loads), then the remainder.
    int ch0 = 0;
    for (; ch0 + 4 <= C; ch0 += 4) {
        cudaError_t e = launch_box_cc<4, false>(g, sidecar, C, ch0, out, resolver, output, stream);
        if (e != cudaSuccess) return e;
    }
    switch (C - ch0) {
        case 1: return launch_box_cc<1, false>(g, sidecar, C, ch0, out, resolver, output, stream);
        case 2: return launch_box_cc<2, false>(g, sidecar, C, ch0, out, resolver, output, stream);
        case 3: return launch_box_cc<3, false>(g, sidecar, C, ch0, out, resolver, output, stream);
        default: return cudaSuccess;
    }
}

cudaError_t launch_box_taps(const DevGrid& g, uint32_t* taps, int resolver, cudaStream_t stream) {
    if (g.n_blocks == 0) return cudaMemsetAsync(taps, 0, sizeof(uint32_t) * kBoxTaps, stream);
    const dim3 grid(g.n_blocks), block(threads_for(g.log2w));
    if (resolver == VBM_RESOLVE_CACHED) box_taps_kernel<true><<<grid, block, 0, stream>>>(g, taps);
    else box_taps_kernel<false><<<grid, block, 0, stream>>>(g, taps);
    return cudaGetLastError();
}

}  // namespace vbm
