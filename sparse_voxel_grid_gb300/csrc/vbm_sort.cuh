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

// Multi-CTA exclusive scan, for arrays of many tiles: tile t covers
// a[t*kScanTile .. (t+1)*kScanTile), one CTA of kScanThreads threads with
// kScanItems consecutive elements per thread.
constexpr int kScanItems = 4;
constexpr uint32_t kScanTile = (uint32_t)kScanThreads * kScanItems;

inline uint32_t scan_tiles(uint64_t n) { return (uint32_t)((n + kScanTile - 1) / kScanTile); }

// Exclusive scan of one value per thread across the CTA; *block_total gets the
// CTA's sum (all threads).
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* warp_sum, uint32_t& block_total) {
    const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= (uint32_t)d) incl += t;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const uint32_t ws = lane < (blockDim.x >> 5) ? warp_sum[lane] : 0u;
        uint32_t wi = ws;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, wi, d);
            if (lane >= (uint32_t)d) wi += t;
        }
        warp_sum[lane] = wi - ws;
        if (lane == 31) warp_sum[32] = wi;
    }
    __syncthreads();
    block_total = warp_sum[32];
    return warp_sum[warp] + incl - v;
}

// sums[t] = sum of tile t.
__global__ void __launch_bounds__(kScanThreads) tile_sum_kernel(const uint32_t* __restrict__ a, uint64_t n,
                                                                 uint32_t* __restrict__ sums) {
    __shared__ uint32_t warp_sum[33];
    const uint64_t i0 = (uint64_t)blockIdx.x * kScanTile + (uint64_t)threadIdx.x * kScanItems;
    uint32_t v = 0;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k)
        if (i0 + k < n) v += a[i0 + k];
    uint32_t total;
    block_exclusive_scan(v, warp_sum, total);
    if (threadIdx.x == 0) sums[blockIdx.x] = total;
}

// a[i] = offs[t] + the exclusive prefix of a within tile t, in place.
__global__ void __launch_bounds__(kScanThreads) tile_scan_kernel(uint32_t* __restrict__ a, uint64_t n,
                                                                  const uint32_t* __restrict__ offs) {
    __shared__ uint32_t warp_sum[33];
    const uint64_t i0 = (uint64_t)blockIdx.x * kScanTile + (uint64_t)threadIdx.x * kScanItems;
    uint32_t v[kScanItems], t = 0;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
        v[k] = i0 + k < n ? a[i0 + k] : 0u;
        t += v[k];
    }
    uint32_t total;
    uint32_t run = offs[blockIdx.x] + block_exclusive_scan(t, warp_sum, total);
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
        if (i0 + k < n) a[i0 + k] = run;
        run += v[k];
    }
}

// Exclusive scan of a[0..n) in place, *total (if not NULL) = the sum.  With
// `tmp` (scan_tiles(n) words of device memory) and more than one tile: per-tile
// sums, a single-CTA scan of the sums, per-tile scans; otherwise one CTA.
inline cudaError_t scan_exclusive(uint32_t* a, uint64_t n, uint32_t* total, uint32_t* tmp, cudaStream_t s) {
    const uint32_t tiles = scan_tiles(n);
    if (!tmp || tiles <= 1) {
        scan_exclusive_kernel<<<1, kScanThreads, 0, s>>>(a, n, total);
        return cudaGetLastError();
    }
    tile_sum_kernel<<<tiles, kScanThreads, 0, s>>>(a, n, tmp);
    scan_exclusive_kernel<<<1, kScanThreads, 0, s>>>(tmp, tiles, total);
    tile_scan_kernel<<<tiles, kScanThreads, 0, s>>>(a, n, tmp);
    return cudaGetLastError();
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
