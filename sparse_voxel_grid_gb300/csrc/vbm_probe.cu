// Measurement probes (include/vbm_probe.h): kernels with the brick box
// filter's launch shape that do nothing, or only the filter's dependent loads,
// to give the filters a measured floor on the same GPU.  Nothing here is part
// of the pipeline's results.
#include <cuda_runtime.h>

#include <string>

#include "../../include/vbm_probe.h"
#include "vbm_device.cuh"
#include "vbm_launch.h"

namespace vbm {
namespace {

// Written only for a value no input holds (a NaN with one particular payload),
// so that the probes' loads cannot be dropped as dead code.
__device__ uint32_t g_probe_sink;
constexpr uint32_t kImpossible = 0x7FBFFFFFu;

__global__ void probe_empty_kernel() {}

__global__ void probe_metadata_kernel(DevGrid g) {
    const uint32_t words = (1u << g.log2w) >> 6, b = blockIdx.x;
    if (threadIdx.x > words) return;
    const uint32_t v = threadIdx.x == words ? __ldg(&g.first_leaf[b])
                                            : (uint32_t)__ldg(&g.jump[(size_t)b * words + threadIdx.x]);
    if (v == kImpossible) g_probe_sink = b;
}

// Lane t < 27 of the first warp: block metadata -> neighbour entry t of the
// block's first leaf -> that leaf's mask word and base index -> one sidecar
// value.  Four dependent loads, as in the brick resolver's build of a brick row.
__global__ void probe_chain_kernel(DevGrid g, const float* __restrict__ sc) {
    const uint32_t t = threadIdx.x, b = blockIdx.x;
    if (t >= 27u) return;
    const uint32_t fl = __ldg(&g.first_leaf[b]);
    uint32_t L = __ldg(&g.nbr[(size_t)fl * kNbrStride + t]);
    if (L == kNone) L = fl;
    const uint32_t w = t & 7u;
    const uint64_t word = __ldg(&g.leaves[L].mask[w]);
    const uint32_t base = __ldg(&g.leaves[L].base[w]);
    const uint32_t idx = word ? base : __ldg(&g.leaves[L].first);
    const float v = __ldg(sc + idx);
    if (__float_as_uint(v) == kImpossible) g_probe_sink = b;
}

}  // namespace

cudaError_t launch_probe(const DevGrid& g, int kind, const float* sidecar, cudaStream_t stream) {
    const unsigned threads = (unsigned)threads_for(g.log2w);
    const size_t smem = brick_box_smem_bytes(g.log2w);
    switch (kind) {
        case VBM_PROBE_EMPTY: probe_empty_kernel<<<g.n_blocks, threads, smem, stream>>>(); break;
        case VBM_PROBE_METADATA: probe_metadata_kernel<<<g.n_blocks, threads, smem, stream>>>(g); break;
        default: probe_chain_kernel<<<g.n_blocks, threads, smem, stream>>>(g, sidecar); break;
    }
    return cudaGetLastError();
}

}  // namespace vbm
