/*
 * CPU oracle for the sparse voxel-grid stencil pipeline.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, obviously correct
 * restatement of what the pipeline computes, used to check the CUDA path.  Only
 * the tests, the smoke check and the benchmark's CPU-baseline leg may load it;
 * the product library never links, imports or calls it, and it shares no code
 * with the product (no headers, helpers, tables or generators).
 *
 * Sources (web pages; cited by title and section):
 *   [2263] OpenVDB PR #2263 "Alternative stencil resolvers for VoxelBlockManager"
 *   [2262] OpenVDB PR #2262 "NanoVDB VBM: Streaming box-stencil"
 *   [2258] OpenVDB PR #2258 "VBM select-based inverse-map decode"
 *
 * Readings of what the pages leave open (the same readings the product
 * implements from its own code):
 *   - Index grid ([2262] "What changed": an Index-Grid resolves a voxel to an
 *     index into a sidecar; index 0 is background, the filter skips it).  Active
 *     voxels get indices 1..N in the depth-first order of a NanoVDB-style tree
 *     (root -> 32^3 upper nodes -> 16^3 lower nodes -> 8^3 leaves): upper nodes
 *     by signed (x>>12, y>>12, z>>12) lexicographically, then the lower-node
 *     slot, then the leaf slot, then the in-leaf offset, each slot x-major.
 *   - In-leaf offset off = (x&7)*64 + (y&7)*8 + (z&7); leaf origin = p & ~7.
 *   - Block b of width W holds indices 1+b*W .. (b+1)*W; slots past N decode to
 *     the sentinels leaf 0xFFFFFFFF, offset 0xFFFF ([2258] "Validation" names the
 *     sentinels without values).
 *   - Box taps in order t = (di+1)*9 + (dj+1)*3 + (dk+1) ([2262] "What changed");
 *     cross taps: the same order restricted to the centre and six faces,
 *     t in {4,10,12,13,14,16,22} (the pages give no cross order).
 *   - Box filter: acc = +0; acc += sidecar[idx*C+ch] for each non-zero tap in tap
 *     order, fp32 round-to-nearest, no reassociation ([2262] "What changed",
 *     "A/B"; [2263] "Measurements").
 *   - Laplacian (the 7-point consumer [2258] "A/B - decode" names): s = +0;
 *     s += face value for each active face in increasing t; out = s - 6*centre
 *     with the product and the difference rounded separately.
 *   - 19-tap WENO consumer ([2258] "A/B - decode" names it, no formula): the
 *     taps are the centre and the voxels 1, 2, 3 steps away along each axis, in
 *     increasing (di,dj,dk) lexicographic order (the box order restricted, as
 *     for the cross).  An inactive tap reads sidecar row 0, the background
 *     value's slot of an index grid.  The value is the Godunov upwind squared
 *     gradient norm of a level set phi at unit spacing, built from fifth-order
 *     WENO one-sided derivatives (Jiang & Shu, J. Comput. Phys. 126, 1996;
 *     Jiang & Peng, SIAM J. Sci. Comput. 21, 2000) with epsilon = 1e-6, all in
 *     fp32 with each operation rounded, in the order written below.
 * Build: g++ -std=c++20 -O2 -ffp-contract=off (no FMA, no fast-math).
 */
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <tuple>
#include <vector>

namespace {

// Depth-first position of a voxel in the 5-4-3 tree, as a tuple compared
// lexicographically: (upper origin x,y,z signed; lower slot; leaf slot; offset).
struct TreeKey {
    int32_t ux, uy, uz;
    uint32_t lower, leaf, off;
};

TreeKey tree_key(int32_t x, int32_t y, int32_t z) {
    TreeKey k;
    k.ux = x >> 12;  // arithmetic shift (C++20): floor(x / 4096)
    k.uy = y >> 12;
    k.uz = z >> 12;
    k.lower = (uint32_t)(((x >> 7) & 31) * 1024 + ((y >> 7) & 31) * 32 + ((z >> 7) & 31));
    k.leaf = (uint32_t)(((x >> 3) & 15) * 256 + ((y >> 3) & 15) * 16 + ((z >> 3) & 15));
    k.off = (uint32_t)((x & 7) * 64 + (y & 7) * 8 + (z & 7));
    return k;
}

bool key_less(const TreeKey& a, const TreeKey& b) {
    return std::tie(a.ux, a.uy, a.uz, a.lower, a.leaf, a.off) <
           std::tie(b.ux, b.uy, b.uz, b.lower, b.leaf, b.off);
}

bool key_equal(const TreeKey& a, const TreeKey& b) {
    return !key_less(a, b) && !key_less(b, a);
}

struct Voxel {
    int32_t x, y, z;
    TreeKey key;
};

// Box tap t <-> offset (di,dj,dk) with t = (di+1)*9 + (dj+1)*3 + (dk+1).
void tap_offset(int t, int& di, int& dj, int& dk) {
    di = t / 9 - 1;
    dj = (t / 3) % 3 - 1;
    dk = t % 3 - 1;
}

const int kCrossTaps[7] = {4, 10, 12, 13, 14, 16, 22};

// 19-tap WENO stencil: offsets in increasing (di,dj,dk) lexicographic order.
const int kWenoOffsets[19][3] = {{-3, 0, 0}, {-2, 0, 0}, {-1, 0, 0}, {0, -3, 0}, {0, -2, 0}, {0, -1, 0}, {0, 0, -3},
                                 {0, 0, -2}, {0, 0, -1}, {0, 0, 0},  {0, 0, 1},  {0, 0, 2},  {0, 0, 3},  {0, 1, 0},
                                 {0, 2, 0},  {0, 3, 0},  {1, 0, 0},  {2, 0, 0},  {3, 0, 0}};

// Fifth-order WENO approximation of a one-sided derivative from five
// consecutive first differences a..e (upwind side first).  Three third-order
// candidates on the sub-stencils (a,b,c), (b,c,d), (c,d,e); smoothness
// indicators s_k; weights alpha_k = gamma_k / (s_k + eps)^2 with the ideal
// weights gamma = 0.1, 0.6, 0.3; result = sum alpha_k q_k / (6 sum alpha_k),
// where q_k is six times the k-th candidate.
float weno5(float a, float b, float c, float d, float e) {
    const float k13_12 = 13.0f / 12.0f;
    const float eps = 1.0e-6f;
    const float t1 = a - 2.0f * b + c;
    const float t2 = a - 4.0f * b + 3.0f * c;
    const float s1 = k13_12 * (t1 * t1) + 0.25f * (t2 * t2);
    const float u1 = b - 2.0f * c + d;
    const float u2 = b - d;
    const float s2 = k13_12 * (u1 * u1) + 0.25f * (u2 * u2);
    const float v1 = c - 2.0f * d + e;
    const float v2 = 3.0f * c - 4.0f * d + e;
    const float s3 = k13_12 * (v1 * v1) + 0.25f * (v2 * v2);
    const float r1 = s1 + eps, r2 = s2 + eps, r3 = s3 + eps;
    const float w1 = 0.1f / (r1 * r1);
    const float w2 = 0.6f / (r2 * r2);
    const float w3 = 0.3f / (r3 * r3);
    const float q1 = 2.0f * a - 7.0f * b + 11.0f * c;
    const float q2 = -b + 5.0f * c + 2.0f * d;
    const float q3 = 2.0f * c + 5.0f * d - e;
    const float num = w1 * q1 + w2 * q2 + w3 * q3;
    const float den = 6.0f * (w1 + w2 + w3);
    return num / den;
}

// Godunov upwind square of the derivative along one axis from the values
// p[0..6] at offsets -3..+3 (p[3] the centre).  minus / plus: the left- and
// right-biased WENO derivatives.  Outside the level set (centre > iso) the
// positive part of minus and the negative part of plus compete, inside the
// opposite parts; the larger square wins.
float godunov_axis(const float (&p)[7], bool outside) {
    float d[6];  // d[k] = p[k+1] - p[k]: differences at offsets -2..+3
    for (int k = 0; k < 6; ++k) d[k] = p[k + 1] - p[k];
    const float minus = weno5(d[0], d[1], d[2], d[3], d[4]);
    const float plus = weno5(d[5], d[4], d[3], d[2], d[1]);
    float lo, hi;
    if (outside) {
        lo = minus > 0.0f ? minus : 0.0f;
        hi = plus < 0.0f ? plus : 0.0f;
    } else {
        lo = minus < 0.0f ? minus : 0.0f;
        hi = plus > 0.0f ? plus : 0.0f;
    }
    const float lo2 = lo * lo, hi2 = hi * hi;
    return lo2 > hi2 ? lo2 : hi2;
}

}  // namespace

struct oracle_grid {
    std::vector<Voxel> vox;  // vox[i-1] is the voxel with index i
};

extern "C" {

// Sorts the active coordinates into tree order; index i is then vox[i-1].
// Returns NULL and sets *status = -1 if a coordinate repeats.
oracle_grid* oracle_create(const int32_t* coords, int64_t n, int* status) {
    oracle_grid* g = new oracle_grid;
    g->vox.resize((size_t)n);
    for (int64_t i = 0; i < n; ++i) {
        Voxel& v = g->vox[(size_t)i];
        v.x = coords[3 * i];
        v.y = coords[3 * i + 1];
        v.z = coords[3 * i + 2];
        v.key = tree_key(v.x, v.y, v.z);
    }
    std::sort(g->vox.begin(), g->vox.end(), [](const Voxel& a, const Voxel& b) { return key_less(a.key, b.key); });
    for (int64_t i = 1; i < n; ++i) {
        if (key_equal(g->vox[(size_t)i - 1].key, g->vox[(size_t)i].key)) {
            delete g;
            if (status) *status = -1;
            return nullptr;
        }
    }
    if (status) *status = 0;
    return g;
}

void oracle_free(oracle_grid* g) { delete g; }

int64_t oracle_count(const oracle_grid* g) { return (int64_t)g->vox.size(); }

// Coordinates in index order: out[3*(i-1) .. 3*(i-1)+2] for index i.
void oracle_coords(const oracle_grid* g, int32_t* out) {
    for (size_t i = 0; i < g->vox.size(); ++i) {
        out[3 * i] = g->vox[i].x;
        out[3 * i + 1] = g->vox[i].y;
        out[3 * i + 2] = g->vox[i].z;
    }
}

// Index of the voxel at (x,y,z): 1..N if active, else 0 (background).
int64_t oracle_index(const oracle_grid* g, int32_t x, int32_t y, int32_t z) {
    TreeKey k = tree_key(x, y, z);
    auto it = std::lower_bound(g->vox.begin(), g->vox.end(), k,
                               [](const Voxel& v, const TreeKey& q) { return key_less(v.key, q); });
    if (it == g->vox.end() || !key_equal(it->key, k)) return 0;
    return (int64_t)(it - g->vox.begin()) + 1;
}

// Leaf ordinals by enumeration: walking the indices in order, the ordinal grows
// by one whenever the leaf origin (p & ~7) changes.  leaf_of[i] is the ordinal
// of index i (leaf_of[0] unused, set to 0xFFFFFFFF); origins (may be NULL)
// receives 3 int32 per leaf.  Returns the number of leaves.
int64_t oracle_leaves(const oracle_grid* g, uint32_t* leaf_of, int32_t* origins) {
    int64_t n = (int64_t)g->vox.size();
    int64_t leaves = 0;
    int32_t px = 0, py = 0, pz = 0;
    if (leaf_of) leaf_of[0] = 0xFFFFFFFFu;
    for (int64_t i = 1; i <= n; ++i) {
        const Voxel& v = g->vox[(size_t)i - 1];
        int32_t ox = v.x & ~7, oy = v.y & ~7, oz = v.z & ~7;
        if (i == 1 || ox != px || oy != py || oz != pz) {
            if (origins) {
                origins[3 * leaves] = ox;
                origins[3 * leaves + 1] = oy;
                origins[3 * leaves + 2] = oz;
            }
            ++leaves;
            px = ox; py = oy; pz = oz;
        }
        if (leaf_of) leaf_of[i] = (uint32_t)(leaves - 1);
    }
    return leaves;
}

// Inverse map by enumeration ([2258] "Summary": slot -> (leaf, voxel offset)).
// nBlocks = ceil(N / W) blocks of W = 2^log2w slots; slot s of block b holds
// index 1 + b*W + s; slots past N get the sentinels.
void oracle_decode(const oracle_grid* g, int log2w, uint32_t* leaf_index, uint16_t* voxel_offset) {
    int64_t n = (int64_t)g->vox.size();
    int64_t W = (int64_t)1 << log2w;
    int64_t nblocks = (n + W - 1) / W;
    std::vector<uint32_t> leaf_of((size_t)n + 1);
    oracle_leaves(g, leaf_of.data(), nullptr);
    for (int64_t slot = 0; slot < nblocks * W; ++slot) {
        int64_t index = 1 + slot;
        if (index > n) {
            leaf_index[slot] = 0xFFFFFFFFu;
            voxel_offset[slot] = 0xFFFF;
        } else {
            leaf_index[slot] = leaf_of[(size_t)index];
            voxel_offset[slot] = (uint16_t)g->vox[(size_t)index - 1].key.off;
        }
    }
}

// Block metadata from its definition ([2263] "Built on the register-decode
// API": the block's first leaf is firstLeafID and it spans 1 + popcount(jumpMap)
// leaves; [2258] "What changed": the leaf owning a slot is found by a popcount
// of the leaf-start bits at or before the slot).  first_leaf[b] is the leaf of
// index 1+b*W; bit s (0 <= s < W) of jump[b*(W/64) + s/64] is set iff s >= 1,
// index 1+b*W+s <= N, and that index is the first index of its leaf.
void oracle_blocks(const oracle_grid* g, int log2w, uint32_t* first_leaf, uint64_t* jump) {
    int64_t n = (int64_t)g->vox.size();
    int64_t W = (int64_t)1 << log2w;
    int64_t words = W / 64;
    int64_t nblocks = (n + W - 1) / W;
    std::vector<uint32_t> leaf_of((size_t)n + 1);
    oracle_leaves(g, leaf_of.data(), nullptr);
    for (int64_t b = 0; b < nblocks; ++b) {
        first_leaf[b] = leaf_of[(size_t)(1 + b * W)];
        for (int64_t w = 0; w < words; ++w) jump[b * words + w] = 0;
        for (int64_t s = 1; s < W; ++s) {
            int64_t index = 1 + b * W + s;
            if (index > n) break;
            if (leaf_of[(size_t)index] != leaf_of[(size_t)index - 1])
                jump[b * words + s / 64] |= (uint64_t)1 << (s % 64);
        }
    }
}

// Stencil taps of the voxels with indices which[0..m) (all 1..N when which is
// NULL, rows 0..N with row 0 zero).  shape 27: the box, taps in order
// t = (di+1)*9+(dj+1)*3+(dk+1); shape 7: the cross, taps {4,10,12,13,14,16,22};
// shape 19: the WENO stencil (kWenoOffsets).
// taps[r*shape + j] = index of the neighbour, 0 if inactive.
int oracle_taps(const oracle_grid* g, int shape, const int64_t* which, int64_t m, uint32_t* taps) {
    if (shape != 27 && shape != 7 && shape != 19) return -1;
    int64_t n = (int64_t)g->vox.size();
    int64_t rows = which ? m : n + 1;
    for (int64_t r = 0; r < rows; ++r) {
        int64_t index = which ? which[r] : r;
        for (int j = 0; j < shape; ++j) {
            uint32_t v = 0;
            if (index >= 1 && index <= n) {
                const Voxel& c = g->vox[(size_t)index - 1];
                int di, dj, dk;
                if (shape == 19) {
                    di = kWenoOffsets[j][0];
                    dj = kWenoOffsets[j][1];
                    dk = kWenoOffsets[j][2];
                } else {
                    tap_offset(shape == 27 ? j : kCrossTaps[j], di, dj, dk);
                }
                v = (uint32_t)oracle_index(g, c.x + di, c.y + dj, c.z + dk);
            }
            taps[r * shape + j] = v;
        }
    }
    return 0;
}

// 27-tap box filter ([2262] "What changed": gather sidecar[index*C+ch] for each
// non-zero tap and accumulate per channel, in tap order).
// out has C floats per row; rows as in oracle_taps.
void oracle_box_filter(const oracle_grid* g, const float* sidecar, int C, const int64_t* which, int64_t m,
                       float* out) {
    int64_t n = (int64_t)g->vox.size();
    int64_t rows = which ? m : n + 1;
    for (int64_t r = 0; r < rows; ++r) {
        int64_t index = which ? which[r] : r;
        for (int ch = 0; ch < C; ++ch) out[r * C + ch] = 0.0f;
        if (index < 1 || index > n) continue;
        const Voxel& c = g->vox[(size_t)index - 1];
        for (int ch = 0; ch < C; ++ch) {
            float acc = 0.0f;
            for (int t = 0; t < 27; ++t) {
                int di, dj, dk;
                tap_offset(t, di, dj, dk);
                int64_t nb = oracle_index(g, c.x + di, c.y + dj, c.z + dk);
                if (nb != 0) acc = acc + sidecar[nb * C + ch];
            }
            out[r * C + ch] = acc;
        }
    }
}

// 7-tap cross consumers.  op 0: Laplacian, s = sum of the active face values
// in increasing tap order, out = s - 6*centre (product and difference rounded
// separately).  op 1: plain sum of the 7 taps in tap order (like the box).
int oracle_cross_filter(const oracle_grid* g, const float* sidecar, int C, int op, const int64_t* which,
                        int64_t m, float* out) {
    if (op != 0 && op != 1) return -1;
    int64_t n = (int64_t)g->vox.size();
    int64_t rows = which ? m : n + 1;
    for (int64_t r = 0; r < rows; ++r) {
        int64_t index = which ? which[r] : r;
        for (int ch = 0; ch < C; ++ch) out[r * C + ch] = 0.0f;
        if (index < 1 || index > n) continue;
        const Voxel& c = g->vox[(size_t)index - 1];
        for (int ch = 0; ch < C; ++ch) {
            float s = 0.0f;
            for (int j = 0; j < 7; ++j) {
                int t = kCrossTaps[j];
                if (op == 0 && t == 13) continue;  // the centre enters below
                int di, dj, dk;
                tap_offset(t, di, dj, dk);
                int64_t nb = oracle_index(g, c.x + di, c.y + dj, c.z + dk);
                if (nb != 0) s = s + sidecar[nb * C + ch];
            }
            if (op == 0) {
                float centre = sidecar[index * C + ch];
                float six_c = 6.0f * centre;
                s = s - six_c;
            }
            out[r * C + ch] = s;
        }
    }
    return 0;
}

// 19-tap WENO consumer: out[r] = the Godunov squared gradient norm of phi at
// the voxel (sum over x, y, z of godunov_axis, added in that order); phi has
// N+1 rows, row 0 the background value that inactive taps read.  Rows as in
// oracle_taps; row 0 and rows outside 1..N are +0.
void oracle_weno_filter(const oracle_grid* g, const float* phi, float iso, const int64_t* which, int64_t m,
                        float* out) {
    int64_t n = (int64_t)g->vox.size();
    int64_t rows = which ? m : n + 1;
    for (int64_t r = 0; r < rows; ++r) {
        int64_t index = which ? which[r] : r;
        out[r] = 0.0f;
        if (index < 1 || index > n) continue;
        const Voxel& c = g->vox[(size_t)index - 1];
        const bool outside = phi[index] > iso;
        float total = 0.0f;
        for (int axis = 0; axis < 3; ++axis) {
            float p[7];
            for (int k = -3; k <= 3; ++k) {
                int q[3] = {0, 0, 0};
                q[axis] = k;
                int64_t nb = oracle_index(g, c.x + q[0], c.y + q[1], c.z + q[2]);
                p[k + 3] = phi[nb];  // nb == 0: the background row
            }
            total = total + godunov_axis(p, outside);
        }
        out[r] = total;
    }
}

}  // extern "C"
