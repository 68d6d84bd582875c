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
// t = (di+1)*9+(dj+1)*3+(dk+1); shape 7: the cross, taps {4,10,12,13,14,16,22}.
// taps[r*shape + j] = index of the neighbour, 0 if inactive.
int oracle_taps(const oracle_grid* g, int shape, const int64_t* which, int64_t m, uint32_t* taps) {
    if (shape != 27 && shape != 7) return -1;
    int64_t n = (int64_t)g->vox.size();
    int64_t rows = which ? m : n + 1;
    for (int64_t r = 0; r < rows; ++r) {
        int64_t index = which ? which[r] : r;
        for (int j = 0; j < shape; ++j) {
            uint32_t v = 0;
            if (index >= 1 && index <= n) {
                const Voxel& c = g->vox[(size_t)index - 1];
                int di, dj, dk;
                tap_offset(shape == 27 ? j : kCrossTaps[j], di, dj, dk);
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

}  // extern "C"
