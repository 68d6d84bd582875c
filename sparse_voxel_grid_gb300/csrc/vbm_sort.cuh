// Device primitives for the device-side builder: a single-CTA exclusive scan
// and a stable LSD radix sort of (uint64 key, uint32 value) pairs, 8-bit
// digits.  Written for this library; used only by vbm_build_dev.cu.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace vbm {
namespace devsort {

constexpr int kScanThreads = 1024;
constexpr int kSortThreads = 256;  // one element per thread per tile
constexpr int kDigits = 256;

// In-place exclusive scan of a[0..n) with one CTA of kScanThreads threads;
// *total receives the sum.  n may be large: the CTA walks it in chunks.
__global__ void __launch_bounds__(kScanThreads) scan_exclusive_kernel(uint32_t* __restrict__ a, uint64_t n,
                                                                       uint32_t* __restrict__ total) {
    __shared__ uint32_t warp_sum[kScanThreads / 32];
    __shared__ uint32_t carry_s;
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    if (tid == 0) carry_s = 0;
    __syncthreads();
    for (uint64_t base = 0; base < n; base += kScanThreads) {
        const uint64_t i = base + tid;
        const uint32_t v = i < n ? a[i] : 0u;
        uint32_t incl = v;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= (uint32_t)d) incl += t;
        }
        if (lane == 31) warp_sum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const uint32_t ws = warp_sum[lane];
            uint32_t wi = ws;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint32_t t = __shfl_up_sync(0xffffffffu, wi, d);
                if (lane >= (uint32_t)d) wi += t;
            }
            warp_sum[lane] = wi - ws;  // exclusive offsets of the warps
        }
        __syncthreads();
        const uint32_t carry = carry_s;
        if (i < n) a[i] = carry + warp_sum[warp] + incl - v;
        __syncthreads();
        if (tid == kScanThreads - 1) carry_s = carry + warp_sum[warp] + incl;
        __syncthreads();
    }
    if (tid == 0 && total) *total = carry_s;
}

// Per-tile digit histogram: hist[d * n_tiles + tile].
__global__ void __launch_bounds__(kSortThreads) radix_hist_kernel(const uint64_t* __restrict__ keys, uint64_t n,
                                                                   int shift, uint32_t n_tiles,
                                                                   uint32_t* __restrict__ hist) {
    __shared__ uint32_t h[kDigits];
    const uint32_t tid = threadIdx.x, tile = blockIdx.x;
    h[tid] = 0;
    __syncthreads();
    const uint64_t i = (uint64_t)tile * kSortThreads + tid;
    if (i < n) atomicAdd(&h[(uint32_t)(keys[i] >> shift) & 255u], 1u);
    __syncthreads();
    hist[(size_t)tid * n_tiles + tile] = h[tid];
}

// Stable scatter: an element goes to offs[d * n_tiles + tile] (the exclusive
// scan of the histograms) + the elements of its digit before it in its tile
// (earlier warps, then earlier lanes).
__global__ void __launch_bounds__(kSortThreads) radix_scatter_kernel(const uint64_t* __restrict__ kin,
                                                                      const uint32_t* __restrict__ vin,
                                                                      uint64_t* __restrict__ kout,
                                                                      uint32_t* __restrict__ vout, uint64_t n,
                                                                      int shift, uint32_t n_tiles,
                                                                      const uint32_t* __restrict__ offs) {
    constexpr int kWarps = kSortThreads / 32;
    __shared__ uint32_t wc[kWarps][kDigits];
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5, tile = blockIdx.x;
    for (uint32_t e = tid; e < (uint32_t)(kWarps * kDigits); e += kSortThreads) (&wc[0][0])[e] = 0;
    __syncthreads();
    const uint64_t i = (uint64_t)tile * kSortThreads + tid;
    const bool valid = i < n;
    const uint64_t key = valid ? kin[i] : 0ull;
    const uint32_t d = valid ? (uint32_t)(key >> shift) & 255u : (uint32_t)kDigits;  // kDigits: no digit
    const uint32_t peers = __match_any_sync(0xffffffffu, d);
    const uint32_t rank = (uint32_t)__popc(peers & ((1u << lane) - 1u));
    if (valid && rank == 0) wc[warp][d] = (uint32_t)__popc(peers);
    __syncthreads();
    if (valid) {
        uint32_t before = 0;
        for (uint32_t w = 0; w < warp; ++w) before += wc[w][d];
        const uint32_t dst = offs[(size_t)d * n_tiles + tile] + before + rank;
        kout[dst] = key;
        vout[dst] = vin[i];
    }
}

}  // namespace devsort
}  // namespace vbm
