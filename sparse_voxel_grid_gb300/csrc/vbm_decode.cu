// Select-based inverse-map decode kernel (OpenVDB PR #2258 "VBM select-based
// inverse-map decode", "What changed"): one thread per output slot; each slot
// ranks itself into its leaf with a jumpMap popcount and finds its voxel by a
// select into the leaf mask through the 9-bit prefix directory.  No shared
// memory, no barrier.  Output is structure-of-arrays: a 32-bit leaf index and
// a 16-bit voxel offset per slot, written coalesced.
#include "vbm_device.cuh"
#include "vbm_launch.h"

namespace vbm {
namespace {

__global__ void __launch_bounds__(512) decode_kernel(DevGrid g, uint32_t* __restrict__ leaf_index,
                                                     uint16_t* __restrict__ voxel_offset) {
    const uint32_t W = 1u << g.log2w;
    const uint32_t b = blockIdx.x;
    const uint64_t* jb = g.jump + (size_t)b * (W >> 6);
    const uint32_t fl = __ldg(&g.first_leaf[b]);
    for (uint32_t s = threadIdx.x; s < W; s += blockDim.x) {
        const uint32_t index = 1u + b * W + s;
        const size_t slot = (size_t)b * W + s;
        if (index > g.n) {
            leaf_index[slot] = kNone;
            voxel_offset[slot] = kNoOffset;
        } else {
            const Slot d = decode_slot(g, fl, jb, s, index);
            leaf_index[slot] = d.leaf;
            voxel_offset[slot] = (uint16_t)d.off;
        }
    }
}

}  // namespace

cudaError_t launch_decode(const DevGrid& g, uint32_t* leaf_index, uint16_t* voxel_offset, cudaStream_t stream) {
    if (g.n_blocks == 0) return cudaSuccess;
    decode_kernel<<<g.n_blocks, threads_for(g.log2w), 0, stream>>>(g, leaf_index, voxel_offset);
    return cudaGetLastError();
}

}  // namespace vbm
