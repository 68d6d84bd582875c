// 19-tap WENO stencil consumer and its raw-tap export.
//
// Sources (web pages; cited by title and section):
//   [2258] OpenVDB PR #2258 "VBM select-based inverse-map decode"
//   [2263] OpenVDB PR #2263 "Alternative stencil resolvers for VoxelBlockManager"
//
// The consumer's arithmetic and tap order are in vbm_weno.cuh: the Godunov
// upwind squared gradient norm of a level set from fifth-order WENO one-sided
// derivatives, an inactive tap reading the background row phi[0].
//
// Resolvers: tree walk, or the cached form through the block's staged 7-entry
// face-neighbour row per spanned leaf (an axial tap at most 3 steps away
// leaves its leaf, if at all, through one face).  The brick resolver stages
// the block's leaves and their face slabs in shared memory (vbm_brick.cu).
#include "vbm_launch.h"
#include "vbm_stencil.cuh"
#include "vbm_weno.cuh"

namespace vbm {

namespace {

// Index of tap j of a decoded voxel.  TABLE: through the staged face row
// (entries as in stage_cross_table: 0 -x, 1 -y, 2 -z, 3 self, 4 +z, 5 +y, 6 +x).
template <bool TABLE>
__device__ __forceinline__ uint32_t weno_tap(const DevGrid& g, const uint32_t* row, uint32_t leaf, int32_t lx,
                                             int32_t ly, int32_t lz, int32_t ox, int32_t oy, int32_t oz, int j) {
    const int a = weno_axis(j), k = weno_step(j);
    const int32_t nx = lx + (a == 0 ? k : 0), ny = ly + (a == 1 ? k : 0), nz = lz + (a == 2 ? k : 0);
    if constexpr (TABLE) {
        const int32_t n = a == 0 ? nx : a == 1 ? ny : nz;
        uint32_t NL = leaf;
        if (n < 0) NL = row[a];
        else if (n > 7) NL = row[6 - a];
        return NL == kNone ? 0u : row_index_at(g.rowrank, NL, pack_off(nx, ny, nz));
    } else {
        (void)row;
        (void)leaf;
        return walk_index(g, ox + nx, oy + ny, oz + nz);
    }
}

// One CTA per VBM block, one thread per slot: decode, resolve the 19 taps,
// gather phi (index 0 reads the background row), evaluate.  TAPS: write the
// raw indices instead.
template <bool CACHED, bool TAPS>
__device__ __forceinline__ void weno_block(const DevGrid& g, const float* __restrict__ phi, float iso,
                                           float* __restrict__ out, uint32_t* __restrict__ taps) {
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
        const int32_t lx = (int32_t)(d.off >> 6), ly = (int32_t)((d.off >> 3) & 7u), lz = (int32_t)(d.off & 7u);
        uint32_t st[kWenoTaps];
        if (CACHED && use_table) {
            const uint32_t* row = table + (d.leaf - fl) * kCrossTaps;
            // Taps 6..12 (z-3 .. z+3) lie in the voxel's z-row: its own leaf's
            // row rank, or the same row of the z neighbour the column leaves
            // through (z < 3: -z, z > 4: +z; never both).
            const uint32_t rr = d.off >> 3;
            const uint2 eo = __ldg(&g.rowrank[(size_t)d.leaf * kRowRanks + rr]);
            const uint32_t Nz = lz < 3 ? row[2] : lz > 4 ? row[4] : kNone;
            uint2 en = make_uint2(0u, 0u);
            if (Nz != kNone) en = __ldg(&g.rowrank[(size_t)Nz * kRowRanks + rr]);
#pragma unroll
            for (int j = 0; j < kWenoTaps; ++j) {
                if (j >= 6 && j <= 12) {
                    const int32_t pos = lz + (j - 9);
                    const uint2 e = (pos & ~7) == 0 ? eo : en;
                    const uint32_t p = (uint32_t)pos & 7u;
                    st[j] = ((e.y >> p) & 1u) ? e.x + (uint32_t)__popc(e.y & ((1u << p) - 1u)) : 0u;
                } else {
                    st[j] = weno_tap<true>(g, row, d.leaf, lx, ly, lz, 0, 0, 0, j);
                }
            }
        } else {
            const LeafRec* r = g.leaves + d.leaf;
            const int32_t ox = __ldg(&r->origin[0]), oy = __ldg(&r->origin[1]), oz = __ldg(&r->origin[2]);
#pragma unroll
            for (int j = 0; j < kWenoTaps; ++j) st[j] = weno_tap<false>(g, nullptr, d.leaf, lx, ly, lz, ox, oy, oz, j);
        }
        if constexpr (TAPS) {
            uint32_t* trow = taps + (size_t)index * kWenoTaps;
#pragma unroll
            for (int j = 0; j < kWenoTaps; ++j) trow[j] = st[j];
        } else {
            float v[kWenoTaps];
#pragma unroll
            for (int j = 0; j < kWenoTaps; ++j) v[j] = __ldg(phi + st[j]);
            out[index] = weno_value(v, iso);
        }
    }
    if (b == 0 && threadIdx.x == 0) {
        if constexpr (TAPS) {
            for (int j = 0; j < kWenoTaps; ++j) taps[j] = 0u;
        } else {
            out[0] = 0.0f;
        }
    }
}

template <bool CACHED, bool TAPS>
__global__ void __launch_bounds__(512) weno_kernel(DevGrid g, const float* __restrict__ phi, float iso,
                                                   float* __restrict__ out, uint32_t* __restrict__ taps) {
    weno_block<CACHED, TAPS>(g, phi, iso, out, taps);
}

// The cached filter held to 40 registers (3 CTAs of 512 threads per SM): free,
// it takes 44 and at W=512 runs 2 CTAs per SM, 8% slower.
template <bool CACHED, bool TAPS>
__global__ void __launch_bounds__(512, 3) weno_kernel_r40(DevGrid g, const float* __restrict__ phi, float iso,
                                                          float* __restrict__ out, uint32_t* __restrict__ taps) {
    weno_block<CACHED, TAPS>(g, phi, iso, out, taps);
}

}  // namespace

cudaError_t launch_weno_filter(const DevGrid& g, const float* phi, float iso, float* out, int resolver,
                               cudaStream_t stream) {
    if (g.n_blocks == 0) return cudaMemsetAsync(out, 0, sizeof(float), stream);
    if (resolver == VBM_RESOLVE_BRICK) return launch_brick_weno(g, phi, iso, out, stream);
    const dim3 grid(g.n_blocks), block(threads_for(g.log2w));
    if (resolver == VBM_RESOLVE_CACHED) weno_kernel_r40<true, false><<<grid, block, 0, stream>>>(g, phi, iso, out, nullptr);
    else weno_kernel<false, false><<<grid, block, 0, stream>>>(g, phi, iso, out, nullptr);
    return cudaGetLastError();
}

cudaError_t launch_weno_taps(const DevGrid& g, uint32_t* taps, int resolver, cudaStream_t stream) {
    if (g.n_blocks == 0) return cudaMemsetAsync(taps, 0, sizeof(uint32_t) * kWenoTaps, stream);
    if (resolver == VBM_RESOLVE_BRICK) return launch_brick_weno_taps(g, taps, stream);
    const dim3 grid(g.n_blocks), block(threads_for(g.log2w));
    if (resolver == VBM_RESOLVE_CACHED) weno_kernel<true, true><<<grid, block, 0, stream>>>(g, nullptr, 0.0f, nullptr, taps);
    else weno_kernel<false, true><<<grid, block, 0, stream>>>(g, nullptr, 0.0f, nullptr, taps);
    return cudaGetLastError();
}

}  // namespace vbm
