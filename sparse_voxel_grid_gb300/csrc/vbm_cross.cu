// 7-tap cross stencil (centre + six faces): Laplacian / 7-tap sum consumers
// and the raw-tap export.
//
// Sources (web pages; cited by title and section):
//   [2263] OpenVDB PR #2263 "Alternative stencil resolvers for VoxelBlockManager"
//   [2258] OpenVDB PR #2258 "VBM select-based inverse-map decode"
//
// Taps j = 0..6 are the box taps t = 4, 10, 12, 13, 14, 16, 22, i.e. offsets
// (-1,0,0), (0,-1,0), (0,0,-1), (0,0,0), (0,0,1), (0,1,0), (1,0,0).  The cross
// resolvers materialise their 7 taps ([2263] "Notes": there is deliberately no
// streaming cross resolver).  The cached form stages a 7-entry neighbour-leaf
// row per spanned leaf (the pages' 16 x 7 table): entry j is the leaf holding
// tap j's position when that position leaves the voxel's leaf, entry 3 the leaf
// itself.  The 7-point Laplacian is named as a consumer in [2258] "A/B -
// decode"; its formula here is s - 6*centre, s = the active face values summed
// in increasing tap order, the product and the difference rounded separately.
#include "vbm_launch.h"
#include "vbm_stencil.cuh"

namespace vbm {
namespace {

// CT > 0: the row stride C is the compile-time CT (and ch0 is 0).
template <int CC, bool VEC, bool CACHED, int OP, int CT>
__global__ void __launch_bounds__(512) cross_filter_kernel(DevGrid g, const float* __restrict__ sc,
                                                           float* __restrict__ out, int C_rt, int ch0_rt) {
    const int C = CT > 0 ? CT : C_rt, ch0 = CT > 0 ? 0 : ch0_rt;
    __shared__ uint32_t table[CACHED ? VBM_MAX_CACHED_LEAVES * kCrossTaps : 1];
    const uint32_t W = 1u << g.log2w, words = W >> 6;
    const uint32_t b = blockIdx.x;
    const uint64_t* jb = g.jump + (size_t)b * words;
    const uint32_t fl = __ldg(&g.first_leaf[b]);
    // One slot per thread (blockDim == W), decoded before the cached table is
    // staged so that the two sets of loads are in flight together.
    const uint32_t s = threadIdx.x, index = 1u + b * W + s;
    const bool valid = s < W && index <= g.n;
    Slot d{0u, 0u};
    if (valid) d = decode_slot(g, fl, jb, s, index);
    bool use_table = false;
    if constexpr (CACHED) {
        const uint32_t span = block_span(jb, words);
        use_table = span <= VBM_MAX_CACHED_LEAVES;
        if (use_table) stage_cross_table(g, fl, span, table);
    }
    if (valid) {
        if (CACHED && use_table) cross_slot<CC, VEC, true, OP>(g, table + (d.leaf - fl) * kCrossTaps, d, index, sc, out, C, ch0);
        else cross_slot<CC, VEC, false, OP>(g, nullptr, d, index, sc, out, C, ch0);
    }
    if (b == 0 && threadIdx.x < (unsigned)CC) out[ch0 + threadIdx.x] = 0.0f;
}

template <bool CACHED>
__global__ void __launch_bounds__(512) cross_taps_kernel(DevGrid g, uint32_t* __restrict__ taps) {
    __shared__ uint32_t table[CACHED ? VBM_MAX_CACHED_LEAVES * kCrossTaps : 1];
    const uint32_t W = 1u << g.log2w, words = W >> 6;
    const uint32_t b = blockIdx.x;
    const uint64_t* jb = g.jump + (size_t)b * words;
    const uint32_t fl = __ldg(&g.first_leaf[b]);
    bool use_table = false;
    if constexpr (CACHED) {
        const uint32_t span = block_span(jb, words);
        use_table = span <= VBM_MAX_CACHED_LEAVES;
        if (use_table) stage_cross_table(g, fl, span, table);
    }
    for (uint32_t s = threadIdx.x; s < W; s += blockDim.x) {
        const uint32_t index = 1u + b * W + s;
        if (index > g.n) break;
        const Slot d = decode_slot(g, fl, jb, s, index);
        uint32_t st[kCrossTaps];
        if (CACHED && use_table) resolve_cross<true>(g, table + (d.leaf - fl) * kCrossTaps, d, st);
        else resolve_cross<false>(g, nullptr, d, st);
        uint32_t* row = taps + (size_t)index * kCrossTaps;
#pragma unroll
        for (int j = 0; j < kCrossTaps; ++j) row[j] = st[j];
    }
    if (b == 0 && threadIdx.x < (unsigned)kCrossTaps) taps[threadIdx.x] = 0u;
}

template <int CC, bool VEC, int CT = 0>
cudaError_t launch_cross_cc(const DevGrid& g, const float* sc, int C, int ch0, float* out, int resolver, int op,
                            cudaStream_t stream) {
    const dim3 grid(g.n_blocks), block(threads_for(g.log2w));
    const bool cached = resolver == VBM_RESOLVE_CACHED;
    if (op == VBM_CROSS_LAPLACIAN) {
        if (cached) cross_filter_kernel<CC, VEC, true, VBM_CROSS_LAPLACIAN, CT><<<grid, block, 0, stream>>>(g, sc, out, C, ch0);
        else cross_filter_kernel<CC, VEC, false, VBM_CROSS_LAPLACIAN, CT><<<grid, block, 0, stream>>>(g, sc, out, C, ch0);
    } else {
        if (cached) cross_filter_kernel<CC, VEC, true, VBM_CROSS_SUM, CT><<<grid, block, 0, stream>>>(g, sc, out, C, ch0);
        else cross_filter_kernel<CC, VEC, false, VBM_CROSS_SUM, CT><<<grid, block, 0, stream>>>(g, sc, out, C, ch0);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_cross_filter(const DevGrid& g, const float* sidecar, int C, float* out, int resolver, int op,
                                cudaStream_t stream) {
    if (g.n_blocks == 0) return cudaMemsetAsync(out, 0, sizeof(float) * (size_t)C, stream);
    switch (C) {
        case 1: return launch_cross_cc<1, false, 1>(g, sidecar, C, 0, out, resolver, op, stream);
        case 2: return launch_cross_cc<2, false, 2>(g, sidecar, C, 0, out, resolver, op, stream);
        case 3: return launch_cross_cc<3, false, 3>(g, sidecar, C, 0, out, resolver, op, stream);
        case 4: return launch_cross_cc<4, true, 4>(g, sidecar, C, 0, out, resolver, op, stream);
        case 8: return launch_cross_cc<8, true, 8>(g, sidecar, C, 0, out, resolver, op, stream);
        case 16: return launch_cross_cc<16, true, 16>(g, sidecar, C, 0, out, resolver, op, stream);
        default: break;
    }
    int ch0 = 0;
    for (; ch0 + 4 <= C; ch0 += 4) {
        cudaError_t e = launch_cross_cc<4, false>(g, sidecar, C, ch0, out, resolver, op, stream);
        if (e != cudaSuccess) return e;
    }
    switch (C - ch0) {
        case 1: return launch_cross_cc<1, false>(g, sidecar, C, ch0, out, resolver, op, stream);
        case 2: return launch_cross_cc<2, false>(g, sidecar, C, ch0, out, resolver, op, stream);
        case 3: return launch_cross_cc<3, false>(g, sidecar, C, ch0, out, resolver, op, stream);
        default: return cudaSuccess;
    }
}

cudaError_t launch_cross_taps(const DevGrid& g, uint32_t* taps, int resolver, cudaStream_t stream) {
    if (g.n_blocks == 0) return cudaMemsetAsync(taps, 0, sizeof(uint32_t) * kCrossTaps, stream);
    const dim3 grid(g.n_blocks), block(threads_for(g.log2w));
    if (resolver == VBM_RESOLVE_CACHED) cross_taps_kernel<true><<<grid, block, 0, stream>>>(g, taps);
    else cross_taps_kernel<false><<<grid, block, 0, stream>>>(g, taps);
    return cudaGetLastError();
}

}  // namespace vbm
