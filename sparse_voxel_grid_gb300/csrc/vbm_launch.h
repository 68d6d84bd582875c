// Kernel launchers called by the C ABI (vbm_api.cu).  Each enqueues work on
// `stream` and returns the launch status; arguments are validated by the caller.
#pragma once

#include <cuda_runtime.h>

#include "vbm_internal.h"

namespace vbm {

cudaError_t launch_decode(const DevGrid& g, uint32_t* leaf_index, uint16_t* voxel_offset, cudaStream_t stream);
cudaError_t launch_sweep_decode(const DevGrid& g, uint32_t* leaf_index, uint16_t* voxel_offset, cudaStream_t stream);

cudaError_t launch_box_filter(const DevGrid& g, const float* sidecar, int C, float* out, int resolver, int output,
                              cudaStream_t stream);

cudaError_t launch_cross_filter(const DevGrid& g, const float* sidecar, int C, float* out, int resolver, int op,
                                cudaStream_t stream);

cudaError_t launch_box_taps(const DevGrid& g, uint32_t* taps, int resolver, cudaStream_t stream);
cudaError_t launch_cross_taps(const DevGrid& g, uint32_t* taps, int resolver, cudaStream_t stream);
cudaError_t launch_weno_filter(const DevGrid& g, const float* phi, float iso, float* out, int resolver,
                               cudaStream_t stream);
cudaError_t launch_weno_taps(const DevGrid& g, uint32_t* taps, int resolver, cudaStream_t stream);

// Brick resolver (vbm_brick.cu).
cudaError_t launch_brick_box(const DevGrid& g, const float* sidecar, int C, float* out, cudaStream_t stream);
// count (1..VBM_MAX_BATCH) box filters; the widths with a compile-time layout
// share one launch, the others are launched one by one.
cudaError_t launch_brick_box_batch(const DevGrid& g, int count, const float* const* sidecars, const int* C,
                                   float* const* outs, cudaStream_t stream);
// Box filters of count sidecars on the device: the brick resolver's batched
// launches, else one launch per sidecar; an empty grid writes row 0 only
// (vbm_host.cu).
cudaError_t launch_box_batch(const DevGrid& g, int count, const float* const* sidecars, const int* C,
                             float* const* outs, int resolver, cudaStream_t stream);
cudaError_t launch_brick_cross(const DevGrid& g, const float* sidecar, int C, float* out, int op, cudaStream_t stream);
cudaError_t launch_brick_taps(const DevGrid& g, uint32_t* taps, int shape, cudaStream_t stream);
cudaError_t launch_brick_weno(const DevGrid& g, const float* phi, float iso, float* out, cudaStream_t stream);
cudaError_t launch_brick_weno_taps(const DevGrid& g, uint32_t* taps, cudaStream_t stream);
// Dynamic shared memory of the brick box/cross kernels at block width 2^log2w.
size_t brick_box_smem_bytes(int log2w);

// Row gather (dst[k] = src[rows[k]]) or scatter (dst[rows[k]] = src[k]) of
// C-float rows (vbm_shard.cu).
cudaError_t launch_rows(bool gather, const float* src, int C, const uint32_t* rows, uint64_t count, float* dst,
                        cudaStream_t stream);

// Measurement probes (vbm_probe.cu, include/vbm_probe.h).
cudaError_t launch_probe(const DevGrid& g, int kind, const float* sidecar, cudaStream_t stream);
// Fills both row-rank tables (kRowRanks) of n_leaves leaf records and their
// neighbour rows (vbm_build_dev.cu).
cudaError_t launch_row_ranks(const LeafRec* leaves, const uint32_t* nbr, uint32_t n_leaves, uint2* rowrank,
                             uint4* rowrank_z, cudaStream_t stream);
// Per-device kernel attributes (shared-memory opt-ins), set once when a grid
// is created on the device, outside any stream capture.
cudaError_t prepare_device_kernels(int device);

// Threads per block for a block width of 2^log2w slots (one slot per thread).
inline int threads_for(int log2w) { return 1 << log2w; }

}  // namespace vbm
