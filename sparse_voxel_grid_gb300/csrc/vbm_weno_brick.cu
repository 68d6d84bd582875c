// 19-tap WENO consumer through bricks (the WENO arithmetic and tap order are
// in vbm_weno.cuh; the per-block decode prologue in vbm_brick.cuh).
//
// Sources (web pages; cited by title and section):
//   [2258] OpenVDB PR #2258 "VBM select-based inverse-map decode"
//   [2263] OpenVDB PR #2263 "Alternative stencil resolvers for VoxelBlockManager"
#include <mutex>

#include "vbm_brick.cuh"
#include "vbm_launch.h"
#include "vbm_weno.cuh"

namespace vbm {
namespace {

using brick::BrickCtx;
using brick::brick_prologue;

// ---------------------------------------------------------------------------
// 19-tap WENO through bricks.  The WENO taps reach 3 steps along one axis, so
// a leaf's brick is a 14x14x14 box (leaf-relative -3..10 on each axis) of
// which only the cells a tap can reach are filled: the 64 core z-rows (x, y in
// 0..7; z in -3..10) and the 48 + 48 rows of the x and y face slabs (one of
// x, y in -3..-1 or 8..10, the other in 0..7; z in 0..7).  Cells hold
// phi[idx] (VALUES; an inactive cell holds phi[0], the background) or idx.
// Only rows whose x lies within 3 of the x range of the block's voxels of that
// leaf are built.
// ---------------------------------------------------------------------------
constexpr int kWEdge = 14;
constexpr int kWCells = kWEdge * kWEdge * kWEdge;
constexpr int kWRows = 64 + 48 + 48;

// Leaves whose WENO bricks are built per round, by block width: about the
// leaves a block spans on the shell (a 64-slot block rarely spans two), within
// shared memory that keeps two 512-thread CTAs per SM.
__host__ __device__ constexpr int weno_group(int log2w) { return log2w <= 6 ? 1 : log2w == 7 ? 2 : log2w == 8 ? 3 : 6; }

__host__ __device__ constexpr size_t weno_smem_bytes(int log2w) {
    return (size_t)weno_group(log2w) * kWCells * sizeof(uint32_t) + (size_t)3 * ((1u << log2w) + 1) * sizeof(uint16_t);
}

__device__ __forceinline__ constexpr int wcell(int x, int y, int z) { return (x + 3) * 196 + (y + 3) * 14 + (z + 3); }

__device__ __forceinline__ constexpr int weno_cell_delta(int j) {
    return weno_axis(j) == 0 ? weno_step(j) * 196 : weno_axis(j) == 1 ? weno_step(j) * 14 : weno_step(j);
}

// Row r of a leaf's WENO brick -> its leaf-relative (x, y).
__device__ __forceinline__ void weno_row_xy(uint32_t r, int& x, int& y) {
    if (r < 64u) {
        x = (int)(r >> 3);
        y = (int)(r & 7u);
    } else if (r < 112u) {
        const int q = (int)(r - 64u), a = q >> 3;
        x = a < 3 ? a - 3 : a + 5;
        y = q & 7;
    } else {
        const int q = (int)(r - 112u), a = q >> 3;
        y = a < 3 ? a - 3 : a + 5;
        x = q & 7;
    }
}

// Indices of leaf L's cells (x&7, y&7, 0..7) (0 where inactive or L is kNone).
__device__ __forceinline__ void row_indices8(const LeafRec* __restrict__ leaves, uint32_t L, int x, int y,
                                             uint32_t (&idx)[8]) {
    uint32_t byte = 0, rb = 0;
    if (L != kNone) {
        const LeafRec* r = leaves + L;
        const uint32_t xw = (uint32_t)(x & 7), yb = (uint32_t)(y & 7) * 8u;
        const uint64_t word = __ldg(&r->mask[xw]);
        byte = (uint32_t)(word >> yb) & 0xFFu;
        rb = __ldg(&r->base[xw]) + (uint32_t)__popcll(word & ((1ull << yb) - 1ull));
    }
#pragma unroll
    for (int z = 0; z < 8; ++z) idx[z] = ((byte >> z) & 1u) ? rb + (uint32_t)__popc(byte & ((1u << z) - 1u)) : 0u;
}

template <bool VALUES>
__device__ __forceinline__ void weno_build_round(const DevGrid& g, const BrickCtx& k, const uint16_t* offs,
                                                 const uint16_t* starts, uint32_t l0, uint32_t nb, uint32_t* wb,
                                                 const float* __restrict__ phi) {
    for (uint32_t e = threadIdx.x; e < nb * (uint32_t)kWRows; e += blockDim.x) {
        const uint32_t kk = e / (uint32_t)kWRows, r = e - kk * (uint32_t)kWRows, l = l0 + kk;
        int x, y;
        weno_row_xy(r, x, y);
        const int x0 = (int)(offs[starts[l]] >> 6), x1 = (int)(offs[starts[l + 1] - 1u] >> 6);
        if (x < x0 - 3 || x > x1 + 3) continue;
        const uint32_t* nrow = g.nbr + (size_t)(k.fl + l) * kNbrStride;
        const int sx = x < 0 ? 0 : x > 7 ? 2 : 1, sy = y < 0 ? 0 : y > 7 ? 2 : 1;
        uint32_t idx[8];
        row_indices8(g.leaves, __ldg(nrow + sx * 9 + sy * 3 + 1), x, y, idx);
        uint32_t* dst = wb + kk * kWCells + wcell(x, y, 0);
        if constexpr (VALUES) {
#pragma unroll
            for (int z = 0; z < 8; ++z) dst[z] = __float_as_uint(__ldg(phi + idx[z]));
        } else {
#pragma unroll
            for (int z = 0; z < 8; ++z) dst[z] = idx[z];
        }
        if (r < 64u) {  // core row: the z halo, 3 cells from each z neighbour
            uint32_t lo[8], hi[8];
            row_indices8(g.leaves, __ldg(nrow + 12), x, y, lo);
            row_indices8(g.leaves, __ldg(nrow + 14), x, y, hi);
            if constexpr (VALUES) {
#pragma unroll
                for (int z = 0; z < 3; ++z) {
                    dst[z - 3] = __float_as_uint(__ldg(phi + lo[5 + z]));
                    dst[8 + z] = __float_as_uint(__ldg(phi + hi[z]));
                }
            } else {
#pragma unroll
                for (int z = 0; z < 3; ++z) {
                    dst[z - 3] = lo[5 + z];
                    dst[8 + z] = hi[z];
                }
            }
        }
    }
    __syncthreads();
}

struct WenoSmem {
    uint32_t* wb;
    uint16_t *offs, *lof, *starts;
    uint32_t group;
};

__device__ __forceinline__ WenoSmem carve_weno(unsigned char* smem, int log2w) {
    WenoSmem m;
    const uint32_t W1 = (1u << log2w) + 1u;
    m.group = (uint32_t)weno_group(log2w);
    m.wb = reinterpret_cast<uint32_t*>(smem);
    m.offs = reinterpret_cast<uint16_t*>(m.wb + m.group * kWCells);
    m.lof = m.offs + W1;
    m.starts = m.lof + W1;
    return m;
}

// TAPS: write the raw indices instead of the WENO value.
template <bool TAPS>
__global__ void __launch_bounds__(512) brick_weno_kernel(DevGrid g, const float* __restrict__ phi, float iso,
                                                         float* __restrict__ out, uint32_t* __restrict__ taps) {
    extern __shared__ __align__(16) unsigned char smem[];
    const WenoSmem m = carve_weno(smem, g.log2w);
    BrickCtx k;
    brick_prologue<true>(g, k, m.offs, m.lof, m.starts, blockIdx.x);
    for (uint32_t l0 = 0; l0 < k.span; l0 += m.group) {
        const uint32_t nb = min(m.group, k.span - l0);
        weno_build_round<!TAPS>(g, k, m.offs, m.starts, l0, nb, m.wb, phi);
        for (uint32_t s = m.starts[l0] + threadIdx.x; s < m.starts[l0 + nb]; s += blockDim.x) {
            const uint32_t* wbk = m.wb + (uint32_t)(m.lof[s] - l0) * kWCells;
            const uint32_t off = m.offs[s];
            const int cc = wcell((int)(off >> 6), (int)((off >> 3) & 7u), (int)(off & 7u));
            const uint32_t index = 1u + k.b * k.W + s;
            if constexpr (TAPS) {
                uint32_t* row = taps + (size_t)index * kWenoTaps;
#pragma unroll
                for (int j = 0; j < kWenoTaps; ++j) row[j] = wbk[cc + weno_cell_delta(j)];
            } else {
                float v[kWenoTaps];
#pragma unroll
                for (int j = 0; j < kWenoTaps; ++j) v[j] = __uint_as_float(wbk[cc + weno_cell_delta(j)]);
                out[index] = weno_value(v, iso);
            }
        }
        __syncthreads();  // the next round overwrites the bricks
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        if constexpr (TAPS) {
            for (int j = 0; j < kWenoTaps; ++j) taps[j] = 0u;
        } else {
            out[0] = 0.0f;
        }
    }
}

}  // namespace

// Dynamic shared memory above the default 48 KB needs an opt-in per kernel
// and device.  It is set when a grid is created (prepare_device_kernels), so
// that a launch is nothing but a launch and can be captured into a CUDA graph.
cudaError_t prepare_device_kernels(int device) {
    static std::mutex mu;
    static uint64_t done = 0;  // one bit per device
    std::lock_guard<std::mutex> lock(mu);
    if (device >= 0 && device < 64 && ((done >> device) & 1u)) return cudaSuccess;
    const int bytes = (int)weno_smem_bytes(9);
    cudaError_t e = cudaFuncSetAttribute(brick_weno_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(brick_weno_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && device >= 0 && device < 64) done |= 1ull << device;
    return e;
}

cudaError_t launch_brick_weno(const DevGrid& g, const float* phi, float iso, float* out, cudaStream_t stream) {
    brick_weno_kernel<false><<<g.n_blocks, threads_for(g.log2w), weno_smem_bytes(g.log2w), stream>>>(g, phi, iso, out,
                                                                                                      nullptr);
    return cudaGetLastError();
}

cudaError_t launch_brick_weno_taps(const DevGrid& g, uint32_t* taps, cudaStream_t stream) {
    brick_weno_kernel<true><<<g.n_blocks, threads_for(g.log2w), weno_smem_bytes(g.log2w), stream>>>(g, nullptr, 0.0f,
                                                                                                     nullptr, taps);
    return cudaGetLastError();
}

}  // namespace vbm
