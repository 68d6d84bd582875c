// Device-side index-grid and VBM-metadata builder (vbm_build_device).
//
// Produces exactly the arrays of the host builder (vbm_build.cpp) from
// coordinates already in device memory, without sorting the voxels:
//   1. leaf origins are inserted into an open-addressing hash table
//      (atomicCAS on 64-bit packed keys) and the occupied slots compacted into
//      provisional leaf ids;
//   2. every voxel sets its bit in its leaf's mask with a 64-bit atomicOr (the
//      returned old word detects duplicates);
//   3. the leaves (not the voxels) are put in depth-first tree order by a
//      stable LSD radix sort of their 54-bit tree keys;
//   4. scans give each leaf's first index and the upper/lower node ids;
//   5. leaf records, child tables, VBM block metadata (firstLeafID, jumpMap)
//      and neighbour rows are filled by one thread per leaf (or per block).
// Temporary device memory is allocated here and freed before returning.
// Coordinates must satisfy |x|,|y|,|z| < 2^20 so that leaf keys fit 54 bits.
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>
#include <string>
#include <vector>

#include "vbm_internal.h"
#include "vbm_launch.h"
#include "vbm_sort.cuh"

namespace vbm {
namespace {

constexpr uint64_t kEmptyKey = ~0ull;
constexpr int32_t kDevCoordLimit = 1 << 20;
constexpr int kThreads = 256;
constexpr uint32_t kBias18 = 1u << 17;  // leaf coordinate (x>>3) + 2^17 fits 18 bits
constexpr uint32_t kBias9 = 1u << 8;    // upper coordinate (x>>12) + 2^8 fits 9 bits

__device__ __forceinline__ uint64_t pack_leaf(int32_t lx, int32_t ly, int32_t lz) {  // lx = x >> 3
    return ((uint64_t)(uint32_t)(lx + (int32_t)kBias18) << 36) | ((uint64_t)(uint32_t)(ly + (int32_t)kBias18) << 18) |
           (uint64_t)(uint32_t)(lz + (int32_t)kBias18);
}
__device__ __forceinline__ void unpack_leaf(uint64_t k, int32_t& lx, int32_t& ly, int32_t& lz) {
    lx = (int32_t)((k >> 36) & 0x3FFFFu) - (int32_t)kBias18;
    ly = (int32_t)((k >> 18) & 0x3FFFFu) - (int32_t)kBias18;
    lz = (int32_t)(k & 0x3FFFFu) - (int32_t)kBias18;
}

// Tree key of a leaf (origin = 8*(lx,ly,lz)): biased upper coordinates (9 bits
// each), then the lower slot (15 bits), then the leaf slot (12 bits).
// Unsigned order = the builder's depth-first order.
__device__ __forceinline__ uint64_t tree_key(int32_t lx, int32_t ly, int32_t lz) {
    const int32_t x = lx * 8, y = ly * 8, z = lz * 8;
    const uint64_t up = ((uint64_t)(uint32_t)((x >> 12) + (int32_t)kBias9) << 18) |
                        ((uint64_t)(uint32_t)((y >> 12) + (int32_t)kBias9) << 9) |
                        (uint64_t)(uint32_t)((z >> 12) + (int32_t)kBias9);
    const uint64_t lower = (uint64_t)(((x >> 7) & 31) << 10 | ((y >> 7) & 31) << 5 | ((z >> 7) & 31));
    const uint64_t leaf = (uint64_t)(((x >> 3) & 15) << 8 | ((y >> 3) & 15) << 4 | ((z >> 3) & 15));
    return (up << 27) | (lower << 12) | leaf;
}

__device__ __forceinline__ uint64_t mix64d(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

// Slot of `key` in the table (inserting it when `insert`; *fresh tells whether
// this call inserted it).  Linear probing from a mixed hash, stopped after
// kMaxProbe slots: a table at most half full ends far sooner.  -1 when the key
// is absent (lookup) or no slot was found (insert).
constexpr uint64_t kMaxProbe = 1u << 12;
__device__ __forceinline__ int64_t probe(uint64_t* keys, uint64_t mask, uint64_t key, bool insert,
                                         bool* fresh = nullptr) {
    uint64_t slot = mix64d(key) & mask;
    for (uint64_t it = 0; it <= mask && it < kMaxProbe; ++it) {
        // A slot only ever changes from empty to a key, so a plain read that
        // shows a key is final; an empty one is settled by the compare-and-swap.
        uint64_t cur = keys[slot];
        if (insert && cur == kEmptyKey)
            cur = atomicCAS((unsigned long long*)&keys[slot], (unsigned long long)kEmptyKey, (unsigned long long)key);
        if (cur == key || (insert && cur == kEmptyKey)) {
            if (fresh) *fresh = insert && cur == kEmptyKey;
            return (int64_t)slot;
        }
        if (!insert && cur == kEmptyKey) return -1;
        slot = (slot + 1) & mask;
    }
    return -1;
}

// 1. Insert leaf keys; flag coordinates out of range (err bit 0) and failed
// probes (bit 1).  With `count`: count the distinct keys and flag (bit 2) a
// table past `limit` keys.
__global__ void insert_kernel(const int32_t* __restrict__ coords, uint64_t n, uint64_t* keys, uint64_t mask,
                              uint32_t* __restrict__ err, uint32_t* __restrict__ count = nullptr,
                              uint32_t limit = 0) {
    // Warp-uniform loop: the lanes of a warp that hold the same leaf key insert
    // it once (the lowest such lane).
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t w0 = blockIdx.x * (uint64_t)blockDim.x + (threadIdx.x & ~31u); w0 < n; w0 += stride) {
        const uint64_t i = w0 + lane;
        uint64_t key = kEmptyKey;
        if (i < n) {
            const int32_t x = coords[3 * i], y = coords[3 * i + 1], z = coords[3 * i + 2];
            if (x <= -kDevCoordLimit || x >= kDevCoordLimit || y <= -kDevCoordLimit || y >= kDevCoordLimit ||
                z <= -kDevCoordLimit || z >= kDevCoordLimit)
                atomicOr(err, 1u);
            else
                key = pack_leaf(x >> 3, y >> 3, z >> 3);
        }
        const uint32_t peers = __match_any_sync(0xffffffffu, key);
        if (key == kEmptyKey || lane != (uint32_t)__ffs(peers) - 1u) continue;
        bool fresh = false;
        if (probe(keys, mask, key, true, &fresh) < 0) atomicOr(err, 2u);
        else if (fresh && count && atomicAdd(count, 1u) >= limit) atomicOr(err, 4u);
    }
}

// 2. Compact occupied slots into provisional leaf ids (arbitrary order).
__global__ void compact_kernel(const uint64_t* __restrict__ keys, uint64_t cap, uint32_t* __restrict__ slot_id,
                               uint32_t* __restrict__ counter, uint64_t* __restrict__ tkey, uint32_t* __restrict__ tval,
                               uint64_t* __restrict__ pkey) {
    for (uint64_t s = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; s < cap; s += (uint64_t)gridDim.x * blockDim.x) {
        const uint64_t k = keys[s];
        if (k == kEmptyKey) continue;
        const uint32_t id = atomicAdd(counter, 1u);
        slot_id[s] = id;
        int32_t lx, ly, lz;
        unpack_leaf(k, lx, ly, lz);
        tkey[id] = tree_key(lx, ly, lz);
        tval[id] = id;
        pkey[id] = k;
    }
}

// 3. Set each voxel's bit in its provisional leaf's mask; count repeats.
__global__ void mask_kernel(const int32_t* __restrict__ coords, uint64_t n, uint64_t* keys, uint64_t mask,
                            const uint32_t* __restrict__ slot_id, unsigned long long* __restrict__ tmask,
                            uint32_t* __restrict__ dups) {
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n; i += (uint64_t)gridDim.x * blockDim.x) {
        const int32_t x = coords[3 * i], y = coords[3 * i + 1], z = coords[3 * i + 2];
        const int64_t slot = probe(keys, mask, pack_leaf(x >> 3, y >> 3, z >> 3), false);
        if (slot < 0) continue;  // reported by insert_kernel
        const uint32_t off = (uint32_t)((x & 7) << 6 | (y & 7) << 3 | (z & 7));
        const unsigned long long bit = 1ull << (off & 63u);
        const unsigned long long old = atomicOr(&tmask[(size_t)slot_id[slot] * 8u + (off >> 6)], bit);
        if (old & bit) atomicAdd(dups, 1u);
    }
}

// 4. Per final leaf: popcount of its mask (input of the first-index scan) and
// the inverse permutation.
__global__ void count_kernel(const uint32_t* __restrict__ perm, uint32_t nl, const unsigned long long* __restrict__ tmask,
                             uint32_t* __restrict__ cnt, uint32_t* __restrict__ final_of) {
    for (uint32_t L = blockIdx.x * blockDim.x + threadIdx.x; L < nl; L += gridDim.x * blockDim.x) {
        const uint32_t t = perm[L];
        uint32_t c = 0;
        for (int w = 0; w < 8; ++w) c += (uint32_t)__popcll(tmask[(size_t)t * 8u + w]);
        cnt[L] = c;
        final_of[t] = L;
    }
}

// Node-boundary flags on the sorted tree keys: upper node changes / lower node changes.
__global__ void node_flag_kernel(const uint64_t* __restrict__ skey, uint32_t nl, uint32_t* __restrict__ up_flag,
                                 uint32_t* __restrict__ lo_flag) {
    for (uint32_t L = blockIdx.x * blockDim.x + threadIdx.x; L < nl; L += gridDim.x * blockDim.x) {
        const uint64_t k = skey[L];
        const bool nu = L == 0 || (skey[L - 1] >> 27) != (k >> 27);
        const bool nlw = L == 0 || (skey[L - 1] >> 12) != (k >> 12);
        up_flag[L] = nu ? 1u : 0u;
        lo_flag[L] = nlw ? 1u : 0u;
    }
}

__global__ void count_occupied_kernel(const uint64_t* __restrict__ keys, uint64_t cap, uint32_t* __restrict__ counter) {
    uint32_t c = 0;
    for (uint64_t s = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; s < cap; s += (uint64_t)gridDim.x * blockDim.x)
        c += keys[s] != kEmptyKey;
    c = __reduce_add_sync(0xffffffffu, c);
    if ((threadIdx.x & 31u) == 0 && c) atomicAdd(counter, c);
}

// 5a. Leaf records in tree order: masks, 9-bit directory, per-word bases, first
// index (1 + exclusive scan of the counts), origin.
__global__ void leafrec_kernel(const uint32_t* __restrict__ perm, uint32_t nl, const unsigned long long* __restrict__ tmask,
                               const uint32_t* __restrict__ cnt_ex, const uint64_t* __restrict__ pkey,
                               LeafRec* __restrict__ leaves) {
    for (uint32_t L = blockIdx.x * blockDim.x + threadIdx.x; L < nl; L += gridDim.x * blockDim.x) {
        const uint32_t t = perm[L];
        LeafRec r;
        const uint32_t first = 1u + cnt_ex[L];
        uint32_t run = 0;
        r.prefix = 0;
        for (int w = 0; w < 8; ++w) {
            r.mask[w] = tmask[(size_t)t * 8u + w];
            if (w >= 1) r.prefix |= (uint64_t)run << (9 * (w - 1));
            r.base[w] = first + run;
            run += (uint32_t)__popcll(r.mask[w]);
        }
        r.first = first;
        r.count = run;
        int32_t lx, ly, lz;
        unpack_leaf(pkey[t], lx, ly, lz);
        r.origin[0] = lx * 8;
        r.origin[1] = ly * 8;
        r.origin[2] = lz * 8;
        r.pad = 0;
        leaves[L] = r;
    }
}

// 5b. Root keys and dense child tables.  up_ex/lo_ex: exclusive scans of the
// node-boundary flags over the sorted tree keys.
__global__ void tables_kernel(const uint64_t* __restrict__ skey, uint32_t nl, const uint32_t* __restrict__ up_ex,
                              const uint32_t* __restrict__ lo_ex, const LeafRec* __restrict__ leaves,
                              uint64_t* __restrict__ root_keys, uint32_t* __restrict__ upper, uint32_t* __restrict__ lower) {
    for (uint32_t L = blockIdx.x * blockDim.x + threadIdx.x; L < nl; L += gridDim.x * blockDim.x) {
        const uint64_t k = skey[L];
        const bool nu = L == 0 || (skey[L - 1] >> 27) != (k >> 27);
        const bool nlw = L == 0 || (skey[L - 1] >> 12) != (k >> 12);
        const uint32_t uid = up_ex[L] + (nu ? 1u : 0u) - 1u;
        const uint32_t lid = lo_ex[L] + (nlw ? 1u : 0u) - 1u;
        const int32_t x = leaves[L].origin[0], y = leaves[L].origin[1], z = leaves[L].origin[2];
        if (nu) root_keys[uid] = root_key_of(x, y, z);
        if (nlw) upper[(size_t)uid * kUpperSlots + (uint32_t)((k >> 12) & 32767u)] = lid;
        lower[(size_t)lid * kLowerSlots + (uint32_t)(k & 4095u)] = L;
    }
}

// 5c. VBM blocks: firstLeafID of every block starting inside leaf L; the
// jumpMap bit of L's first index unless it starts a block.
__global__ void blocks_kernel(const LeafRec* __restrict__ leaves, uint32_t nl, int log2w, uint32_t* __restrict__ first_leaf,
                              unsigned long long* __restrict__ jump) {
    const uint32_t W = 1u << log2w, words = W >> 6;
    for (uint32_t L = blockIdx.x * blockDim.x + threadIdx.x; L < nl; L += gridDim.x * blockDim.x) {
        const uint32_t f = leaves[L].first, c = leaves[L].count;  // indices f .. f+c-1
        for (uint32_t b = (f - 1u + W - 1u) >> log2w; (b << log2w) + 1u <= f + c - 1u; ++b) first_leaf[b] = L;
        const uint32_t b = (f - 1u) >> log2w, s = (f - 1u) & (W - 1u);
        if (L > 0 && s != 0) atomicOr(&jump[(size_t)b * words + (s >> 6)], 1ull << (s & 63u));
    }
}

// 5d. Neighbour rows: leaf at origin + 8*(dx,dy,dz), through the hash table.
__global__ void nbr_kernel(const LeafRec* __restrict__ leaves, uint32_t nl, uint64_t* keys, uint64_t mask,
                           const uint32_t* __restrict__ slot_id, const uint32_t* __restrict__ final_of,
                           uint32_t* __restrict__ nbr) {
    const uint64_t total = (uint64_t)nl * kNbrStride;
    for (uint64_t e = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; e < total; e += (uint64_t)gridDim.x * blockDim.x) {
        const uint32_t L = (uint32_t)(e / kNbrStride), t = (uint32_t)(e % kNbrStride);
        uint32_t id = kNone;
        if (t < 27u) {
            const int32_t lx = (leaves[L].origin[0] >> 3) + (int32_t)(t / 9u) - 1;
            const int32_t ly = (leaves[L].origin[1] >> 3) + (int32_t)((t / 3u) % 3u) - 1;
            const int32_t lz = (leaves[L].origin[2] >> 3) + (int32_t)(t % 3u) - 1;
            const int32_t lim = (int32_t)kBias18;
            if (lx >= -lim && lx < lim && ly >= -lim && ly < lim && lz >= -lim && lz < lim) {
                const int64_t slot = probe(keys, mask, pack_leaf(lx, ly, lz), false);
                if (slot >= 0) id = final_of[slot_id[slot]];
            }
        }
        nbr[e] = id;
    }
}

// 5e. Spans: max and the number of blocks over MaxCachedLeaves.
// Index of in-leaf bit `bit` (0..511) of leaf L, 0 if L is absent or the bit clear.
__device__ __forceinline__ uint32_t index_of_bit(const LeafRec* __restrict__ leaves, uint32_t L, uint32_t bit) {
    if (L == kNone) return 0u;
    const uint64_t word = leaves[L].mask[bit >> 6];
    const uint32_t b = bit & 63u;
    return ((word >> b) & 1ull) ? leaves[L].base[bit >> 6] + (uint32_t)__popcll(word & ((1ull << b) - 1ull)) : 0u;
}

// Row ranks, with and without the z halo (kRowRanks): one (leaf, row) entry
// per thread, grid-stride.  The z neighbours come from the leaf's neighbour row
// (slots 12 and 14: offsets (0,0,-1) and (0,0,+1)).
__global__ void rowrank_kernel(const LeafRec* __restrict__ leaves, const uint32_t* __restrict__ nbr, uint32_t nl,
                               uint2* __restrict__ rowrank, uint4* __restrict__ rowrank_z) {
    const uint64_t total = (uint64_t)nl * kRowRanks, stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t e = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += stride) {
        const uint32_t L = (uint32_t)(e >> 6), xy = (uint32_t)e & 63u;  // xy = x*8 + y
        const LeafRec& r = leaves[L];
        const uint32_t x = xy >> 3, shift = 8u * (xy & 7u);
        const uint64_t word = r.mask[x];
        const uint32_t first = r.base[x] + (uint32_t)__popcll(word & ((1ull << shift) - 1ull));
        const uint32_t bits = (uint32_t)(word >> shift) & 0xFFu;
        const uint32_t Lm = nbr[(size_t)L * kNbrStride + 12], Lp = nbr[(size_t)L * kNbrStride + 14];
        rowrank[e] = make_uint2(first, bits);
        rowrank_z[e] = make_uint4(first, bits, index_of_bit(leaves, Lm, xy * 8u + 7u), index_of_bit(leaves, Lp, xy * 8u));
    }
}

__global__ void span_kernel(const unsigned long long* __restrict__ jump, uint32_t n_blocks, uint32_t words,
                            uint32_t* __restrict__ out) {
    for (uint32_t b = blockIdx.x * blockDim.x + threadIdx.x; b < n_blocks; b += gridDim.x * blockDim.x) {
        uint32_t span = 1;
        for (uint32_t w = 0; w < words; ++w) span += (uint32_t)__popcll(jump[(size_t)b * words + w]);
        atomicMax(&out[0], span);
        if (span > VBM_MAX_CACHED_LEAVES) atomicAdd(&out[1], 1u);
    }
}

}  // namespace

namespace {

// The builder's scratch memory comes from a stream-ordered pool of its own,
// one per device, which keeps up to kPoolKeep bytes between builds: a build
// after the first allocates and frees without cudaMalloc / cudaFree (which
// synchronise the device).  The grid's own arena is a plain cudaMalloc.
constexpr uint64_t kPoolKeep = 2ull << 30;

cudaError_t scratch_pool(int device, cudaMemPool_t* out) {
    static std::mutex mu;
    static cudaMemPool_t pools[64] = {};
    if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!pools[device]) {
        cudaMemPoolProps props{};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = device;
        cudaMemPool_t p;
        cudaError_t e = cudaMemPoolCreate(&p, &props);
        if (e != cudaSuccess) return e;
        uint64_t keep = kPoolKeep;
        e = cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep);
        if (e != cudaSuccess) {
            cudaMemPoolDestroy(p);
            return e;
        }
        pools[device] = p;
    }
    *out = pools[device];
    return cudaSuccess;
}

// Device allocations from the pool, freed (stream-ordered) on scope exit.
struct Scratch {
    cudaMemPool_t pool = nullptr;
    cudaStream_t stream = nullptr;
    std::vector<void*> ptrs;
    ~Scratch() {
        for (void* p : ptrs) cudaFreeAsync(p, stream);
    }
    template <typename T>
    cudaError_t alloc(T** p, size_t count) {
        void* q = nullptr;
        const cudaError_t e = cudaMallocFromPoolAsync(&q, count ? count * sizeof(T) : sizeof(T), pool, stream);
        if (e == cudaSuccess) ptrs.push_back(q);
        *p = static_cast<T*>(q);
        return e;
    }
};

unsigned grid_for(uint64_t work, int sm_count) {
    const uint64_t want = (work + kThreads - 1) / kThreads;
    const uint64_t cap = (uint64_t)(sm_count > 0 ? sm_count : 1) * 32u;
    return (unsigned)(want < 1 ? 1 : (want < cap ? want : cap));
}

// Stable radix sort of (key, value) pairs by the low `bits` bits of the keys;
// the result ends in (k0, v0).
cudaError_t radix_sort(uint64_t* k0, uint32_t* v0, uint64_t* k1, uint32_t* v1, uint32_t* hist, uint32_t* scan_tmp,
                       uint32_t n, int bits, cudaStream_t s) {
    const uint32_t tiles = (n + devsort::kSortThreads - 1) / devsort::kSortThreads;
    for (int shift = 0; shift < bits; shift += 8) {
        devsort::radix_hist_kernel<<<tiles, devsort::kSortThreads, 0, s>>>(k0, n, shift, tiles, hist);
        devsort::scan_exclusive(hist, (uint64_t)tiles * devsort::kDigits, nullptr, scan_tmp, s);
        devsort::radix_scatter_kernel<<<tiles, devsort::kSortThreads, 0, s>>>(k0, v0, k1, v1, n, shift, tiles, hist);
        std::swap(k0, k1);
        std::swap(v0, v1);
    }
    // An odd number of passes leaves the result in the second buffers.
    if (((bits + 7) / 8) & 1) {
        cudaMemcpyAsync(k1, k0, (size_t)n * sizeof(uint64_t), cudaMemcpyDeviceToDevice, s);
        cudaMemcpyAsync(v1, v0, (size_t)n * sizeof(uint32_t), cudaMemcpyDeviceToDevice, s);
    }
    return cudaGetLastError();
}

template <typename T>
cudaError_t read_back(T* host, const T* dev, size_t count, cudaStream_t s) {
    cudaError_t e = cudaMemcpyAsync(host, dev, count * sizeof(T), cudaMemcpyDeviceToHost, s);
    return e != cudaSuccess ? e : cudaStreamSynchronize(s);
}

}  // namespace

int build_device(const int32_t* coords, uint64_t n, int log2w, uint32_t flags, void* stream_v, vbm_grid* g,
                 std::string& err) {
    const cudaStream_t st = static_cast<cudaStream_t>(stream_v);
#define VBM_CK(call)                                                                              \
    do {                                                                                          \
        const cudaError_t e_ = (call);                                                            \
        if (e_ != cudaSuccess) {                                                                  \
            cudaGetLastError();                                                                   \
            err = std::string("vbm_build_device: ") + #call + ": " + cudaGetErrorString(e_);      \
            return e_ == cudaErrorMemoryAllocation ? VBM_ERR_NOMEM : VBM_ERR_CUDA;                \
        }                                                                                         \
    } while (0)
    if (n >= (uint64_t)1 << 31) {
        err = "vbm_build_device: N must be < 2^31";
        return VBM_ERR_RANGE;
    }
    int device = 0, sm = 1;
    VBM_CK(cudaGetDevice(&device));
    VBM_CK(cudaDeviceGetAttribute(&sm, cudaDevAttrMultiProcessorCount, device));
    const uint32_t W = 1u << log2w, words = W >> 6;
    Scratch sc;
    sc.stream = st;
    VBM_CK(scratch_pool(device, &sc.pool));

    // 1-2. Leaf hash table and compaction.  The table is first sized for one
    // leaf per 16 voxels (power of two, at most half full); a grid with more
    // leaves than that is rebuilt once in a table of 2n slots, which no input
    // can fill past half.
    uint64_t full = 1024;
    while (full < 2 * n) full <<= 1;
    uint64_t cap = 1024;
    while (cap < 2 * (n / 16 + 1024)) cap <<= 1;
    if (cap > full) cap = full;
    uint64_t* keys;
    uint32_t *slot_id, *ctr;  // ctr: [0] error flags, [1] leaves, [2] repeats, [3..4] span stats, [5..7] totals
    VBM_CK(sc.alloc(&ctr, 8));
    uint32_t h[2];
    for (;;) {
        VBM_CK(sc.alloc(&keys, cap));
        VBM_CK(sc.alloc(&slot_id, cap));
        VBM_CK(cudaMemsetAsync(keys, 0xFF, cap * sizeof(uint64_t), st));
        VBM_CK(cudaMemsetAsync(ctr, 0, 8 * sizeof(uint32_t), st));
        if (n) insert_kernel<<<grid_for(n, sm), kThreads, 0, st>>>(coords, n, keys, cap - 1, ctr, ctr + 1,
                                                                   (uint32_t)(cap / 2));
        VBM_CK(cudaGetLastError());
        VBM_CK(read_back(h, ctr, 2, st));
        if ((h[0] & 4u) && cap < full) {
            cap = full;  // more leaves than the first table holds
            continue;
        }
        break;
    }
    if (h[0] & 1u) {
        err = "vbm_build_device: a coordinate is outside (-2^20, 2^20)";
        return VBM_ERR_RANGE;
    }
    if (h[0] & 2u) {
        err = "vbm_build_device: hash table overflow";
        return VBM_ERR_CUDA;
    }
    const uint32_t nl = h[1];
    uint64_t *tkey, *tkey2, *pkey;
    uint32_t *tval, *tval2, *hist, *cnt, *final_of, *up_f, *lo_f;
    unsigned long long* tmask;
    const uint32_t tiles = (nl + devsort::kSortThreads - 1) / devsort::kSortThreads;
    VBM_CK(sc.alloc(&tkey, nl));
    VBM_CK(sc.alloc(&tkey2, nl));
    VBM_CK(sc.alloc(&pkey, nl));
    VBM_CK(sc.alloc(&tval, nl));
    VBM_CK(sc.alloc(&tval2, nl));
    VBM_CK(sc.alloc(&hist, (size_t)tiles * devsort::kDigits));
    VBM_CK(sc.alloc(&cnt, nl));
    VBM_CK(sc.alloc(&final_of, nl));
    VBM_CK(sc.alloc(&up_f, nl));
    VBM_CK(sc.alloc(&lo_f, nl));
    VBM_CK(sc.alloc(&tmask, (size_t)nl * 8u));
    uint32_t* scan_tmp;  // tile sums of the multi-CTA scans
    VBM_CK(sc.alloc(&scan_tmp, devsort::scan_tiles(std::max<uint64_t>(nl, (uint64_t)tiles * devsort::kDigits)) + 1u));
    VBM_CK(cudaMemsetAsync(ctr + 1, 0, sizeof(uint32_t), st));
    VBM_CK(cudaMemsetAsync(tmask, 0, (size_t)nl * 8u * sizeof(uint64_t), st));
    compact_kernel<<<grid_for(cap, sm), kThreads, 0, st>>>(keys, cap, slot_id, ctr + 1, tkey, tval, pkey);
    // 3. Masks and repeats.
    if (n) mask_kernel<<<grid_for(n, sm), kThreads, 0, st>>>(coords, n, keys, cap - 1, slot_id, tmask, ctr + 2);
    VBM_CK(cudaGetLastError());
    uint32_t dups = 0;
    VBM_CK(read_back(&dups, ctr + 2, 1, st));
    if (dups && !(flags & VBM_BUILD_DEDUP)) {
        err = "vbm_build_device: duplicate coordinates (" + std::to_string(dups) + " repeats)";
        return VBM_ERR_DUPLICATE;
    }
    // 4. Tree order of the leaves; counts, first indices, node ids.
    if (nl) {
        VBM_CK(radix_sort(tkey, tval, tkey2, tval2, hist, scan_tmp, nl, 54, st));
        count_kernel<<<grid_for(nl, sm), kThreads, 0, st>>>(tval, nl, tmask, cnt, final_of);
        node_flag_kernel<<<grid_for(nl, sm), kThreads, 0, st>>>(tkey, nl, up_f, lo_f);
        VBM_CK(devsort::scan_exclusive(cnt, nl, ctr + 5, scan_tmp, st));
        VBM_CK(devsort::scan_exclusive(up_f, nl, ctr + 6, scan_tmp, st));
        VBM_CK(devsort::scan_exclusive(lo_f, nl, ctr + 7, scan_tmp, st));
    }
    uint32_t tot[3] = {0, 0, 0};
    if (nl) VBM_CK(read_back(tot, ctr + 5, 3, st));
    const uint64_t N = tot[0];
    g->n = N;
    g->log2w = log2w;
    g->n_leaves = nl;
    g->n_upper = tot[1];
    g->n_lower = tot[2];
    g->n_blocks = (N + W - 1) / W;
    g->device = device;

    // 5. The grid's arena, laid out as vbm_build's.
    const ArenaLayout lay = arena_layout(nl, g->n_upper, g->n_lower, g->n_blocks, log2w);
    VBM_CK(cudaMalloc(&g->arena, lay.total));
    g->arena_bytes = lay.total;
    char* base = static_cast<char*>(g->arena);
    LeafRec* leaves = reinterpret_cast<LeafRec*>(base + lay.off[0]);
    uint64_t* root_keys = reinterpret_cast<uint64_t*>(base + lay.off[1]);
    uint32_t* upper = reinterpret_cast<uint32_t*>(base + lay.off[2]);
    uint32_t* lower = reinterpret_cast<uint32_t*>(base + lay.off[3]);
    uint32_t* first_leaf = reinterpret_cast<uint32_t*>(base + lay.off[4]);
    unsigned long long* jump = reinterpret_cast<unsigned long long*>(base + lay.off[5]);
    uint32_t* nbr = reinterpret_cast<uint32_t*>(base + lay.off[6]);
    VBM_CK(cudaMemsetAsync(upper, 0xFF, lay.bytes[2], st));
    VBM_CK(cudaMemsetAsync(lower, 0xFF, lay.bytes[3], st));
    VBM_CK(cudaMemsetAsync(jump, 0, lay.bytes[5], st));
    VBM_CK(cudaMemsetAsync(ctr + 3, 0, 2 * sizeof(uint32_t), st));
    if (nl) {
        leafrec_kernel<<<grid_for(nl, sm), kThreads, 0, st>>>(tval, nl, tmask, cnt, pkey, leaves);
        tables_kernel<<<grid_for(nl, sm), kThreads, 0, st>>>(tkey, nl, up_f, lo_f, leaves, root_keys, upper, lower);
        blocks_kernel<<<grid_for(nl, sm), kThreads, 0, st>>>(leaves, nl, log2w, first_leaf, jump);
        nbr_kernel<<<grid_for((uint64_t)nl * kNbrStride, sm), kThreads, 0, st>>>(leaves, nl, keys, cap - 1, slot_id,
                                                                                 final_of, nbr);
        rowrank_kernel<<<grid_for((uint64_t)nl * kRowRanks, sm), kThreads, 0, st>>>(
            leaves, nbr, nl, reinterpret_cast<uint2*>(base + lay.off[7]), reinterpret_cast<uint4*>(base + lay.off[8]));
        span_kernel<<<grid_for(g->n_blocks, sm), kThreads, 0, st>>>(jump, (uint32_t)g->n_blocks, words, ctr + 3);
        VBM_CK(cudaGetLastError());
    }
    uint32_t spans[2] = {0, 0};
    VBM_CK(read_back(spans, ctr + 3, 2, st));
    g->max_span = spans[0];
    g->n_over_cache = spans[1];
    set_device_views(g, lay, sm);
    VBM_CK(prepare_device_kernels(device));
    g->mirrors_filled = false;  // host copies are made on the first vbm_leaf_export
#undef VBM_CK
    return VBM_OK;
}


// ---------------------------------------------------------------------------
// Allocation-free variant.  For callers that cannot call cudaMalloc: all
// temporary memory lives in one file-scope static device array, sized for at
// most kNoAllocMaxVoxels voxels, and the grid's arrays go into the caller's
// buffer.  Every GPU that loads the library holds the static array until the
// process exits.  Calls share it, so calls that overlap on the GPU race.
// ---------------------------------------------------------------------------
namespace {

constexpr uint64_t kNoAllocMaxVoxels = 65536;  // also the most leaves
constexpr uint64_t kNoAllocCap = 2 * kNoAllocMaxVoxels;  // hash capacity (a power of two)

struct NoAllocLayout {
    size_t ctr, keys, slot_id, tkey, tkey2, pkey, tval, tval2, cnt, final_of, up_f, lo_f, hist, tmask, total;
};

constexpr size_t up256(size_t v) { return (v + 255) / 256 * 256; }

constexpr NoAllocLayout noalloc_layout() {
    NoAllocLayout l{};
    size_t o = 0;
    l.ctr = o; o = up256(o + 8 * sizeof(uint32_t));
    l.keys = o; o = up256(o + kNoAllocCap * sizeof(uint64_t));
    l.slot_id = o; o = up256(o + kNoAllocCap * sizeof(uint32_t));
    l.tkey = o; o = up256(o + kNoAllocMaxVoxels * sizeof(uint64_t));
    l.tkey2 = o; o = up256(o + kNoAllocMaxVoxels * sizeof(uint64_t));
    l.pkey = o; o = up256(o + kNoAllocMaxVoxels * sizeof(uint64_t));
    l.tval = o; o = up256(o + kNoAllocMaxVoxels * sizeof(uint32_t));
    l.tval2 = o; o = up256(o + kNoAllocMaxVoxels * sizeof(uint32_t));
    l.cnt = o; o = up256(o + kNoAllocMaxVoxels * sizeof(uint32_t));
    l.final_of = o; o = up256(o + kNoAllocMaxVoxels * sizeof(uint32_t));
    l.up_f = o; o = up256(o + kNoAllocMaxVoxels * sizeof(uint32_t));
    l.lo_f = o; o = up256(o + kNoAllocMaxVoxels * sizeof(uint32_t));
    l.hist = o; o = up256(o + kNoAllocMaxVoxels * sizeof(uint32_t));  // 256 digits x kNoAllocMaxVoxels/256 tiles
    l.tmask = o; o = up256(o + 8 * kNoAllocMaxVoxels * sizeof(uint64_t));
    l.total = o;
    return l;
}

constexpr NoAllocLayout kNoAlloc = noalloc_layout();

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAlloc.total];

// Device address of the static scratch array, looked up once per device with
// that device current.  The lookup and the table are guarded by one mutex, so
// first calls on the same device from several host threads are safe; a failed
// lookup leaves the entry empty and is retried by the next call.
constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

cudaError_t noalloc_scratch(int device, unsigned char** out) {
    if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[device]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_noalloc_ptr[device] = p;
    }
    *out = static_cast<unsigned char*>(g_noalloc_ptr[device]);
    return cudaSuccess;
}

}  // namespace

int build_device_noalloc(const int32_t* coords, uint64_t n, int log2w, uint32_t flags, void* arena,
                         uint64_t arena_bytes, uint64_t* arena_needed, void* stream_v, vbm_grid* g, std::string& err) {
    const cudaStream_t st = static_cast<cudaStream_t>(stream_v);
#define VBM_CK(call)                                                                                  \
    do {                                                                                              \
        const cudaError_t e_ = (call);                                                                \
        if (e_ != cudaSuccess) {                                                                      \
            cudaGetLastError();                                                                       \
            err = std::string("vbm_build_device_noalloc: ") + #call + ": " + cudaGetErrorString(e_);  \
            return VBM_ERR_CUDA;                                                                      \
        }                                                                                             \
    } while (0)
    if (arena_needed) *arena_needed = 0;
    if (n > kNoAllocMaxVoxels) {
        err = "vbm_build_device_noalloc: " + std::to_string(n) + " voxels exceed the maximum of " +
              std::to_string(kNoAllocMaxVoxels) + " that its static scratch memory holds";
        return VBM_ERR_RANGE;
    }
    if (((uintptr_t)arena & 255u) != 0) {
        err = "vbm_build_device_noalloc: arena must be 256-byte aligned";
        return VBM_ERR_ALIGN;
    }
    int device = 0, sm = 1;
    VBM_CK(cudaGetDevice(&device));
    VBM_CK(cudaDeviceGetAttribute(&sm, cudaDevAttrMultiProcessorCount, device));
    unsigned char* base_s = nullptr;
    VBM_CK(noalloc_scratch(device, &base_s));
    const uint32_t W = 1u << log2w, words = W >> 6;
    uint32_t* ctr = reinterpret_cast<uint32_t*>(base_s + kNoAlloc.ctr);
    uint64_t* keys = reinterpret_cast<uint64_t*>(base_s + kNoAlloc.keys);
    uint32_t* slot_id = reinterpret_cast<uint32_t*>(base_s + kNoAlloc.slot_id);
    uint64_t* tkey = reinterpret_cast<uint64_t*>(base_s + kNoAlloc.tkey);
    uint64_t* tkey2 = reinterpret_cast<uint64_t*>(base_s + kNoAlloc.tkey2);
    uint64_t* pkey = reinterpret_cast<uint64_t*>(base_s + kNoAlloc.pkey);
    uint32_t* tval = reinterpret_cast<uint32_t*>(base_s + kNoAlloc.tval);
    uint32_t* tval2 = reinterpret_cast<uint32_t*>(base_s + kNoAlloc.tval2);
    uint32_t* cnt = reinterpret_cast<uint32_t*>(base_s + kNoAlloc.cnt);
    uint32_t* final_of = reinterpret_cast<uint32_t*>(base_s + kNoAlloc.final_of);
    uint32_t* up_f = reinterpret_cast<uint32_t*>(base_s + kNoAlloc.up_f);
    uint32_t* lo_f = reinterpret_cast<uint32_t*>(base_s + kNoAlloc.lo_f);
    uint32_t* hist = reinterpret_cast<uint32_t*>(base_s + kNoAlloc.hist);
    unsigned long long* tmask = reinterpret_cast<unsigned long long*>(base_s + kNoAlloc.tmask);

    // The array keeps the previous call's contents: clear what must start empty.
    uint64_t cap = 1024;
    while (cap < 2 * n) cap <<= 1;
    VBM_CK(cudaMemsetAsync(ctr, 0, 8 * sizeof(uint32_t), st));
    VBM_CK(cudaMemsetAsync(keys, 0xFF, cap * sizeof(uint64_t), st));
    if (n) insert_kernel<<<grid_for(n, sm), kThreads, 0, st>>>(coords, n, keys, cap - 1, ctr);
    count_occupied_kernel<<<grid_for(cap, sm), kThreads, 0, st>>>(keys, cap, ctr + 1);
    VBM_CK(cudaGetLastError());
    uint32_t h[2];
    VBM_CK(read_back(h, ctr, 2, st));
    if (h[0] & 1u) {
        err = "vbm_build_device_noalloc: a coordinate is outside (-2^20, 2^20)";
        return VBM_ERR_RANGE;
    }
    if (h[0] & 2u) {
        err = "vbm_build_device_noalloc: hash table overflow";
        return VBM_ERR_CUDA;
    }
    const uint32_t nl = h[1];
    VBM_CK(cudaMemsetAsync(ctr + 1, 0, sizeof(uint32_t), st));
    VBM_CK(cudaMemsetAsync(tmask, 0, (size_t)nl * 8u * sizeof(uint64_t), st));
    compact_kernel<<<grid_for(cap, sm), kThreads, 0, st>>>(keys, cap, slot_id, ctr + 1, tkey, tval, pkey);
    if (n) mask_kernel<<<grid_for(n, sm), kThreads, 0, st>>>(coords, n, keys, cap - 1, slot_id, tmask, ctr + 2);
    VBM_CK(cudaGetLastError());
    uint32_t dups = 0;
    VBM_CK(read_back(&dups, ctr + 2, 1, st));
    if (dups && !(flags & VBM_BUILD_DEDUP)) {
        err = "vbm_build_device_noalloc: duplicate coordinates (" + std::to_string(dups) + " repeats)";
        return VBM_ERR_DUPLICATE;
    }
    if (nl) {
        VBM_CK(radix_sort(tkey, tval, tkey2, tval2, hist, nullptr, nl, 54, st));
        count_kernel<<<grid_for(nl, sm), kThreads, 0, st>>>(tval, nl, tmask, cnt, final_of);
        node_flag_kernel<<<grid_for(nl, sm), kThreads, 0, st>>>(tkey, nl, up_f, lo_f);
        devsort::scan_exclusive_kernel<<<1, devsort::kScanThreads, 0, st>>>(cnt, nl, ctr + 5);
        devsort::scan_exclusive_kernel<<<1, devsort::kScanThreads, 0, st>>>(up_f, nl, ctr + 6);
        devsort::scan_exclusive_kernel<<<1, devsort::kScanThreads, 0, st>>>(lo_f, nl, ctr + 7);
        VBM_CK(cudaGetLastError());
    }
    uint32_t tot[3] = {0, 0, 0};
    if (nl) VBM_CK(read_back(tot, ctr + 5, 3, st));
    const uint64_t N = tot[0];
    const uint64_t n_blocks = (N + W - 1) / W;
    const ArenaLayout lay = arena_layout(nl, tot[1], tot[2], n_blocks, log2w);
    if (arena_needed) *arena_needed = lay.total;
    // lay.total is at least 256 bytes (arena_layout), so a NULL arena is always
    // too small, also for an empty grid.
    if (arena_bytes < lay.total || !arena) {
        err = "vbm_build_device_noalloc: the arena holds " + std::to_string(arena_bytes) + " bytes; this grid needs " +
              std::to_string(lay.total);
        return VBM_ERR_RANGE;
    }
    g->n = N;
    g->log2w = log2w;
    g->n_leaves = nl;
    g->n_upper = tot[1];
    g->n_lower = tot[2];
    g->n_blocks = n_blocks;
    g->device = device;
    g->arena = arena;
    g->arena_bytes = lay.total;
    g->owns_arena = false;
    g->host_mirrors = false;
    char* base = static_cast<char*>(arena);
    LeafRec* leaves = reinterpret_cast<LeafRec*>(base + lay.off[0]);
    uint64_t* root_keys = reinterpret_cast<uint64_t*>(base + lay.off[1]);
    uint32_t* upper = reinterpret_cast<uint32_t*>(base + lay.off[2]);
    uint32_t* lower = reinterpret_cast<uint32_t*>(base + lay.off[3]);
    uint32_t* first_leaf = reinterpret_cast<uint32_t*>(base + lay.off[4]);
    unsigned long long* jump = reinterpret_cast<unsigned long long*>(base + lay.off[5]);
    uint32_t* nbr = reinterpret_cast<uint32_t*>(base + lay.off[6]);
    VBM_CK(cudaMemsetAsync(upper, 0xFF, lay.bytes[2], st));
    VBM_CK(cudaMemsetAsync(lower, 0xFF, lay.bytes[3], st));
    VBM_CK(cudaMemsetAsync(jump, 0, lay.bytes[5], st));
    VBM_CK(cudaMemsetAsync(ctr + 3, 0, 2 * sizeof(uint32_t), st));
    if (nl) {
        leafrec_kernel<<<grid_for(nl, sm), kThreads, 0, st>>>(tval, nl, tmask, cnt, pkey, leaves);
        tables_kernel<<<grid_for(nl, sm), kThreads, 0, st>>>(tkey, nl, up_f, lo_f, leaves, root_keys, upper, lower);
        blocks_kernel<<<grid_for(nl, sm), kThreads, 0, st>>>(leaves, nl, log2w, first_leaf, jump);
        nbr_kernel<<<grid_for((uint64_t)nl * kNbrStride, sm), kThreads, 0, st>>>(leaves, nl, keys, cap - 1, slot_id,
                                                                                 final_of, nbr);
        rowrank_kernel<<<grid_for((uint64_t)nl * kRowRanks, sm), kThreads, 0, st>>>(
            leaves, nbr, nl, reinterpret_cast<uint2*>(base + lay.off[7]), reinterpret_cast<uint4*>(base + lay.off[8]));
        span_kernel<<<grid_for(n_blocks, sm), kThreads, 0, st>>>(jump, (uint32_t)n_blocks, words, ctr + 3);
        VBM_CK(cudaGetLastError());
    }
    uint32_t spans[2] = {0, 0};
    VBM_CK(read_back(spans, ctr + 3, 2, st));
    g->max_span = spans[0];
    g->n_over_cache = spans[1];
    set_device_views(g, lay, sm);
    VBM_CK(prepare_device_kernels(device));
#undef VBM_CK
    return VBM_OK;
}

cudaError_t launch_row_ranks(const LeafRec* leaves, const uint32_t* nbr, uint32_t n_leaves, uint2* rowrank,
                             uint4* rowrank_z, cudaStream_t stream) {
    if (!n_leaves) return cudaSuccess;
    int device = 0, sm = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sm, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) return e;
    rowrank_kernel<<<grid_for((uint64_t)n_leaves * kRowRanks, sm), kThreads, 0, stream>>>(leaves, nbr, n_leaves, rowrank,
                                                                                          rowrank_z);
    return cudaGetLastError();
}

}  // namespace vbm
