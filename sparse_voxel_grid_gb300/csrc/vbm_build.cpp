// Host-side index-grid and VBM-metadata builder.
//
// The pages do not describe how the grid is built (NanoVDB builds it); this
// builder produces the structures the decode and the resolvers read:
//   - 8^3 leaves with 512-bit value masks and the 9-bit per-word prefix-sum
//     directory (OpenVDB PR #2258 "VBM select-based inverse-map decode",
//     "Summary": the leaf's 9-bit mPrefixSum guides the select),
//   - upper tree levels (root table -> 32^3 upper -> 16^3 lower -> leaf) for
//     the root-down walk (PR #2263 "Alternative stencil resolvers for
//     VoxelBlockManager", "Summary"),
//   - consecutive indices 1..N in depth-first tree order, and
//   - per-block firstLeafID / jumpMap (PR #2263, "Built on the register-decode
//     API": the block's first leaf is firstLeafID and it spans
//     1 + popcount(jumpMap) leaves).
// O(N) pass over the coordinates (leaf hash table), then a sort of the leaves.
#include <algorithm>
#include <cstring>
#include <numeric>

#include "vbm_internal.h"

namespace vbm {
namespace {

constexpr int32_t kCoordLimit = 1 << 30;

uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

// Open-addressing hash table: leaf origin -> provisional leaf id.
class LeafTable {
   public:
    explicit LeafTable(size_t expect) { rehash(std::max<size_t>(64, next_pow2(expect * 2))); }

    // Returns the id of the leaf at (x,y,z), inserting `fresh` if absent.
    uint32_t find_or_insert(int32_t x, int32_t y, int32_t z, uint32_t fresh, bool& inserted) {
        if ((size_ + 1) * 2 > cap_) rehash(cap_ * 2);
        size_t h = slot_of(x, y, z);
        for (;;) {
            uint32_t id = ids_[h];
            if (id == kNone) {
                ids_[h] = fresh;
                keys_[3 * h] = x; keys_[3 * h + 1] = y; keys_[3 * h + 2] = z;
                ++size_;
                inserted = true;
                return fresh;
            }
            if (keys_[3 * h] == x && keys_[3 * h + 1] == y && keys_[3 * h + 2] == z) {
                inserted = false;
                return id;
            }
            h = (h + 1) & (cap_ - 1);
        }
    }

    // Id of the leaf at (x,y,z), or kNone.
    uint32_t find(int32_t x, int32_t y, int32_t z) const {
        size_t h = slot_of(x, y, z);
        for (;;) {
            uint32_t id = ids_[h];
            if (id == kNone) return kNone;
            if (keys_[3 * h] == x && keys_[3 * h + 1] == y && keys_[3 * h + 2] == z) return id;
            h = (h + 1) & (cap_ - 1);
        }
    }

   private:
    static size_t next_pow2(size_t v) {
        size_t p = 1;
        while (p < v) p <<= 1;
        return p;
    }
    size_t slot_of(int32_t x, int32_t y, int32_t z) const {
        uint64_t k = ((uint64_t)(uint32_t)x * 0x9E3779B97F4A7C15ULL) ^ ((uint64_t)(uint32_t)y << 21) ^
                     ((uint64_t)(uint32_t)z * 0xC2B2AE3D27D4EB4FULL);
        return (size_t)mix64(k) & (cap_ - 1);
    }
    void rehash(size_t cap) {
        std::vector<int32_t> ok = std::move(keys_);
        std::vector<uint32_t> oi = std::move(ids_);
        size_t ocap = cap_;
        cap_ = cap;
        keys_.assign(3 * cap_, 0);
        ids_.assign(cap_, kNone);
        size_ = 0;
        for (size_t i = 0; i < ocap; ++i) {
            if (oi[i] == kNone) continue;
            size_t h = slot_of(ok[3 * i], ok[3 * i + 1], ok[3 * i + 2]);
            while (ids_[h] != kNone) h = (h + 1) & (cap_ - 1);
            ids_[h] = oi[i];
            keys_[3 * h] = ok[3 * i]; keys_[3 * h + 1] = ok[3 * i + 1]; keys_[3 * h + 2] = ok[3 * i + 2];
            ++size_;
        }
    }
    std::vector<int32_t> keys_;
    std::vector<uint32_t> ids_;
    size_t cap_ = 0, size_ = 0;
};

inline uint32_t lower_slot_of(int32_t x, int32_t y, int32_t z) {
    return (uint32_t)(((x >> 7) & 31) << 10 | ((y >> 7) & 31) << 5 | ((z >> 7) & 31));
}
inline uint32_t leaf_slot_of(int32_t x, int32_t y, int32_t z) {
    return (uint32_t)(((x >> 3) & 15) << 8 | ((y >> 3) & 15) << 4 | ((z >> 3) & 15));
}

}  // namespace

int build_host(const int32_t* coords, uint64_t n, int log2w, uint32_t flags, vbm_grid* g, std::string& err) {
    if (n >= (uint64_t)1 << 31) {
        err = "vbm_build: N must be < 2^31";
        return VBM_ERR_RANGE;
    }
    const uint64_t W = (uint64_t)1 << log2w;
    const int words = (int)(W / 64);

    // 1. Provisional leaves: origin and mask, in order of first appearance.
    std::vector<int32_t> p_origin;
    std::vector<uint64_t> p_mask;
    LeafTable table(n / 64 + 16);
    uint64_t dups = 0;
    for (uint64_t i = 0; i < n; ++i) {
        int32_t x = coords[3 * i], y = coords[3 * i + 1], z = coords[3 * i + 2];
        if (x < -kCoordLimit || x > kCoordLimit || y < -kCoordLimit || y > kCoordLimit || z < -kCoordLimit ||
            z > kCoordLimit) {
            err = "vbm_build: coordinate " + std::to_string(i) + " outside [-2^30, 2^30]";
            return VBM_ERR_RANGE;
        }
        bool inserted = false;
        uint32_t id = table.find_or_insert(x & ~7, y & ~7, z & ~7, (uint32_t)(p_origin.size() / 3), inserted);
        if (inserted) {
            p_origin.push_back(x & ~7);
            p_origin.push_back(y & ~7);
            p_origin.push_back(z & ~7);
            p_mask.resize(p_mask.size() + 8, 0);
        }
        uint32_t off = (uint32_t)((x & 7) << 6 | (y & 7) << 3 | (z & 7));
        uint64_t& word = p_mask[(size_t)id * 8 + (off >> 6)];
        uint64_t bit = (uint64_t)1 << (off & 63);
        if (word & bit) {
            if (!(flags & VBM_BUILD_DEDUP)) {
                err = "vbm_build: duplicate coordinate (" + std::to_string(x) + "," + std::to_string(y) + "," +
                      std::to_string(z) + ")";
                return VBM_ERR_DUPLICATE;
            }
            ++dups;
        }
        word |= bit;
    }
    const uint64_t N = n - dups;
    const size_t nl = p_origin.size() / 3;

    // 2. Leaves in depth-first tree order: root key, then lower slot, then leaf slot.
    std::vector<uint64_t> k_root(nl), k_low(nl);
    for (size_t l = 0; l < nl; ++l) {
        int32_t x = p_origin[3 * l], y = p_origin[3 * l + 1], z = p_origin[3 * l + 2];
        k_root[l] = root_key_of(x, y, z);
        k_low[l] = (uint64_t)lower_slot_of(x, y, z) << 12 | leaf_slot_of(x, y, z);
    }
    std::vector<uint32_t> order(nl);
    std::iota(order.begin(), order.end(), 0u);
    std::sort(order.begin(), order.end(), [&](uint32_t a, uint32_t b) {
        return k_root[a] != k_root[b] ? k_root[a] < k_root[b] : k_low[a] < k_low[b];
    });

    // 3. Leaf records: counts, first indices, 9-bit directory, per-word bases.
    g->n = N;
    g->log2w = log2w;
    g->n_leaves = nl;
    g->leaves.assign(nl, LeafRec{});
    uint32_t next_index = 1;
    for (size_t l = 0; l < nl; ++l) {
        const uint32_t src = order[l];
        LeafRec& r = g->leaves[l];
        std::memset(&r, 0, sizeof(r));
        uint32_t run = 0;
        r.prefix = 0;
        for (int w = 0; w < 8; ++w) {
            r.mask[w] = p_mask[(size_t)src * 8 + w];
            if (w >= 1) r.prefix |= (uint64_t)run << (9 * (w - 1));
            r.base[w] = next_index + run;
            run += (uint32_t)__builtin_popcountll(r.mask[w]);
        }
        r.first = next_index;
        r.count = run;
        r.origin[0] = p_origin[3 * src];
        r.origin[1] = p_origin[3 * src + 1];
        r.origin[2] = p_origin[3 * src + 2];
        next_index += run;
    }

    // 4. Tree levels.  Upper nodes = distinct root keys (sorted); lower nodes =
    //    distinct (root key, lower slot) in leaf order.
    g->root_keys.clear();
    std::vector<uint32_t> leaf_upper(nl), leaf_lower(nl);
    uint32_t n_lower = 0;
    for (size_t l = 0; l < nl; ++l) {
        const uint32_t src = order[l];
        if (g->root_keys.empty() || g->root_keys.back() != k_root[src]) g->root_keys.push_back(k_root[src]);
        leaf_upper[l] = (uint32_t)g->root_keys.size() - 1;
        bool new_lower = l == 0 || k_root[order[l - 1]] != k_root[src] ||
                         (k_low[order[l - 1]] >> 12) != (k_low[src] >> 12);
        if (new_lower) ++n_lower;
        leaf_lower[l] = n_lower - 1;
    }
    g->n_upper = (uint32_t)g->root_keys.size();
    g->n_lower = n_lower;
    g->upper.assign((size_t)g->n_upper * kUpperSlots, kNone);
    g->lower.assign((size_t)g->n_lower * kLowerSlots, kNone);
    for (size_t l = 0; l < nl; ++l) {
        const uint32_t src = order[l];
        uint32_t lower_slot = (uint32_t)(k_low[src] >> 12), leaf_slot = (uint32_t)(k_low[src] & 4095);
        g->upper[(size_t)leaf_upper[l] * kUpperSlots + lower_slot] = leaf_lower[l];
        g->lower[(size_t)leaf_lower[l] * kLowerSlots + leaf_slot] = (uint32_t)l;
    }

    // 5. VBM blocks: firstLeafID = leaf of index 1+b*W; jumpMap bit s set iff
    //    index 1+b*W+s (s >= 1) is the first index of a leaf.
    g->n_blocks = (N + W - 1) / W;
    g->first_leaf.assign(g->n_blocks, 0);
    g->jump.assign(g->n_blocks * (size_t)words, 0);
    size_t L = 0;
    for (uint64_t b = 0; b < g->n_blocks; ++b) {
        uint64_t i0 = 1 + b * W;
        while (L + 1 < nl && g->leaves[L + 1].first <= i0) ++L;
        g->first_leaf[b] = (uint32_t)L;
    }
    for (size_t l = 1; l < nl; ++l) {
        uint64_t f = g->leaves[l].first;
        uint64_t b = (f - 1) / W, s = (f - 1) % W;
        if (s != 0) g->jump[b * words + s / 64] |= (uint64_t)1 << (s % 64);
    }
    // 6. Neighbour rows: nbr[L*32 + (dx+1)*9 + (dy+1)*3 + (dz+1)] = id of the leaf
    //    at origin(L) + 8*(dx,dy,dz), or kNone; entries 27..31 are padding.  The
    //    GB300 brick resolver reads these instead of probing the tree per block.
    {
        LeafTable final_ids(nl + 16);
        for (size_t l = 0; l < nl; ++l) {
            bool ins = false;
            final_ids.find_or_insert(g->leaves[l].origin[0], g->leaves[l].origin[1], g->leaves[l].origin[2],
                                     (uint32_t)l, ins);
        }
        g->nbr.assign(nl * kNbrStride, kNone);
        for (size_t l = 0; l < nl; ++l) {
            const int32_t* o = g->leaves[l].origin;
            for (int t = 0; t < 27; ++t) {
                const int32_t x = o[0] + 8 * (t / 9 - 1), y = o[1] + 8 * ((t / 3) % 3 - 1), z = o[2] + 8 * (t % 3 - 1);
                g->nbr[l * kNbrStride + t] = final_ids.find(x, y, z);
            }
        }
    }
    g->n_over_cache = 0;
    g->max_span = 0;
    for (uint64_t b = 0; b < g->n_blocks; ++b) {
        uint32_t span = 1;
        for (int w = 0; w < words; ++w) span += (uint32_t)__builtin_popcountll(g->jump[b * words + w]);
        g->max_span = std::max(g->max_span, span);
        if (span > VBM_MAX_CACHED_LEAVES) ++g->n_over_cache;
    }
    return VBM_OK;
}

}  // namespace vbm
