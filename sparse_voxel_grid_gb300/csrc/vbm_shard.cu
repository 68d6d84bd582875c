// Block-range shards (include/vbm.h, "Block-range shards"): the halo of a
// shard, computed on the host from the grid's arrays, and the row gather /
// scatter kernels that pack and place the exchanged sidecar rows.
//
// Source (web page; cited by title and section):
//   [2263] OpenVDB PR #2263 "Alternative stencil resolvers for VoxelBlockManager"
//   ("Summary": a block's voxels span few distinct, consecutive leaves, which
//   is what makes a contiguous block range a compact shard).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <vector>

#include "vbm_internal.h"
#include "vbm_launch.h"

namespace vbm {

// Sorted indices outside the shard's own range [1 + b0*W, min(N, b1*W)] of the
// active voxels of every neighbour leaf (27 per leaf, the builder's rows) of
// every leaf the blocks b0 .. b1-1 span.  Any box or cross tap of a voxel of
// leaf L lies in one of L's 27 neighbour leaves, so these rows are all the
// shard reads beyond its own.  The grid's host arrays must be filled.
void shard_halo(const vbm_grid* g, uint32_t b0, uint32_t b1, std::vector<uint32_t>& rows) {
    rows.clear();
    if (b0 >= b1) return;
    const uint32_t W = 1u << g->log2w, words = W >> 6;
    const uint64_t lo = 1 + (uint64_t)b0 * W, hi = std::min<uint64_t>(g->n, (uint64_t)b1 * W);
    const uint32_t L_first = g->first_leaf[b0];
    uint32_t L_last = g->first_leaf[b1 - 1];
    for (uint32_t w = 0; w < words; ++w) L_last += (uint32_t)__builtin_popcountll(g->jump[(size_t)(b1 - 1) * words + w]);
    std::vector<uint32_t> nb;
    nb.reserve((size_t)(L_last - L_first + 1) * 8);
    for (uint32_t L = L_first; L <= L_last; ++L)
        for (int t = 0; t < kBoxTaps; ++t) {
            const uint32_t M = g->nbr[(size_t)L * kNbrStride + t];
            if (M != kNone) nb.push_back(M);
        }
    std::sort(nb.begin(), nb.end());
    nb.erase(std::unique(nb.begin(), nb.end()), nb.end());
    // Leaves are numbered in index order, so increasing leaf ids give
    // increasing, disjoint index ranges.
    for (const uint32_t M : nb) {
        const uint64_t f = g->leaves[M].first, e = f + g->leaves[M].count;  // indices f .. e-1
        for (uint64_t i = f; i < std::min(e, lo); ++i) rows.push_back((uint32_t)i);
        for (uint64_t i = std::max(f, hi + 1); i < e; ++i) rows.push_back((uint32_t)i);
    }
}

namespace {

// dst[k*C + c] = src[rows[k]*C + c] (GATHER) or dst[rows[k]*C + c] =
// src[k*C + c], one element per thread of a grid-stride loop.
template <bool GATHER>
__global__ void __launch_bounds__(256) rows_kernel(const float* __restrict__ src, int C,
                                                   const uint32_t* __restrict__ rows, uint64_t count,
                                                   float* __restrict__ dst) {
    const uint64_t total = count * (uint64_t)C;
    for (uint64_t e = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (uint64_t)gridDim.x * blockDim.x) {
        const uint64_t k = e / (uint64_t)C, c = e - k * (uint64_t)C;
        const uint64_t r = (uint64_t)__ldg(&rows[k]) * (uint64_t)C + c;
        if constexpr (GATHER) dst[e] = __ldg(&src[r]);
        else dst[r] = __ldg(&src[e]);
    }
}

}  // namespace

cudaError_t launch_rows(bool gather, const float* src, int C, const uint32_t* rows, uint64_t count, float* dst,
                        cudaStream_t stream) {
    if (count == 0) return cudaSuccess;
    int device = 0, sms = 1;
    cudaError_t e = cudaGetDevice(&device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) return e;
    const uint64_t total = count * (uint64_t)C;
    const uint64_t want = (total + 255) / 256;
    const unsigned grid = (unsigned)std::min<uint64_t>(want, (uint64_t)sms * 8u);
    if (gather) rows_kernel<true><<<grid, 256, 0, stream>>>(src, C, rows, count, dst);
    else rows_kernel<false><<<grid, 256, 0, stream>>>(src, C, rows, count, dst);
    return cudaGetLastError();
}

}  // namespace vbm
