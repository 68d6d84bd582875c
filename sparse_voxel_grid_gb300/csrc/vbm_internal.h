// Internal layout of a vbm_grid: host-side arrays written by the builder and
// the device arena the kernels read.  Shared by the builder (vbm_build.cpp),
// the C ABI (vbm_api.cu) and the kernels; not part of the public interface.
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>
#include <string>
#include <vector>

#include <vector_types.h>

#include "../../include/vbm.h"

#ifdef __CUDACC__
#define VBM_HD __host__ __device__ __forceinline__
#else
#define VBM_HD inline
#endif

namespace vbm {

constexpr uint32_t kNone = 0xFFFFFFFFu;     // absent child / leaf / sentinel leaf index
constexpr uint16_t kNoOffset = 0xFFFF;      // sentinel voxel offset
constexpr int kUpperSlots = 32 * 32 * 32;   // children of an upper node (lower nodes)
constexpr int kLowerSlots = 16 * 16 * 16;   // children of a lower node (leaves)
constexpr int kBoxTaps = 27;
constexpr int kCrossTaps = 7;
constexpr int kWenoTaps = 19;
constexpr int kMaxC = 64;
constexpr int kNbrStride = 32;              // neighbour-row stride: 27 ids + 5 pad = one 128-byte line
// Row ranks: entry L*64 + x*8 + y describes the z-row (x, y, 0..7) of leaf L:
// .y = its 8 mask bits (bit z = voxel (x,y,z) active), .x = the index the
// row's first active voxel has or would have (the leaf's first index plus the
// active voxels before the row in leaf order).  A finer copy of the leaf's
// rank directory, derived from the masks on the device after every build.
// rowrank_z holds the same rows with their z halo, 16 bytes each: .x, .y as
// above, .z = the index of (x, y, -1), i.e. voxel (x,y,7) of the -z neighbour
// leaf, .w = the index of (x, y, 8), voxel (x,y,0) of the +z neighbour (0 where
// that voxel is inactive or its leaf absent), so that one load ranks a whole
// three-tap z column.
constexpr int kRowRanks = 64;

// One leaf: 128 bytes, one cache line.  `mask` is the 512-bit value mask (bit
// off%64 of word off/64, off = x*64 + y*8 + z in-leaf); `prefix` is the 9-bit
// directory the decode reads (field w-1, w = 1..7, at bits 9(w-1)..9w-1 = set
// bits in words 0..w-1); `base[w]` = first + prefix(w) is the same directory
// pre-added to the first index, which the resolvers use to rank a bit with one
// popcount.
struct alignas(128) LeafRec {
    uint64_t mask[8];   // bytes 0..63
    uint32_t base[8];   // bytes 64..95
    uint64_t prefix;    // bytes 96..103
    uint32_t first;     // bytes 104..107: index of the first active voxel
    int32_t origin[3];  // bytes 108..119
    uint32_t count;     // bytes 120..123: active voxels in the leaf
    uint32_t pad;
};
static_assert(sizeof(LeafRec) == 128, "LeafRec must be one 128-byte line");

// Root key of the upper node containing (x,y,z): the signed upper-node
// coordinates (x>>12, y>>12, z>>12) biased by 2^19 into 20 bits each, so that
// unsigned order of keys is signed lexicographic order of the upper origins.
VBM_HD uint64_t root_key_of(int32_t x, int32_t y, int32_t z) {
    return ((uint64_t)(uint32_t)((x >> 12) + (1 << 19)) << 40) | ((uint64_t)(uint32_t)((y >> 12) + (1 << 19)) << 20) |
           (uint64_t)(uint32_t)((z >> 12) + (1 << 19));
}

// Everything a kernel needs, passed by value.
struct DevGrid {
    const LeafRec* leaves;
    const uint64_t* root_keys;   // n_upper sorted keys
    const uint32_t* upper;       // n_upper x 32768: lower-node id or kNone
    const uint32_t* lower;       // n_lower x 4096: leaf id or kNone
    const uint32_t* first_leaf;  // n_blocks
    const uint64_t* jump;        // n_blocks x (W/64)
    const uint32_t* nbr;         // n_leaves x kNbrStride: neighbour-leaf ids (see vbm_build.cpp)
    const uint2* rowrank;        // n_leaves x 64: row ranks of each leaf (see kRowRanks)
    const uint4* rowrank_z;      // n_leaves x 64: the same rows with their z halo (see kRowRanks)
    uint32_t n;                  // active voxels
    uint32_t n_leaves;
    uint32_t n_blocks;           // blocks a launch covers (CTAs of a one-CTA-per-block kernel)
    uint32_t n_upper;
    int log2w;
    int sm_count;                // SMs of the grid's device (for one-wave launches)
    uint32_t block0;             // first block a launch covers: CTA i filters block block0 + i
                                 // (0 for whole-grid calls; a shard's first block otherwise)
};

// Device staging and streams of vbm_box_filter_batch_host (vbm_host.cu).
struct HostIO;
void destroy_host_io(HostIO* h);

}  // namespace vbm

struct vbm_grid {
    // sizes
    uint64_t n = 0;
    int log2w = 7;
    uint32_t n_upper = 0, n_lower = 0;
    uint64_t n_leaves = 0, n_blocks = 0;
    uint64_t n_over_cache = 0;
    uint32_t max_span = 0;
    // host arrays
    std::vector<vbm::LeafRec> leaves;
    std::vector<uint64_t> root_keys;
    std::vector<uint32_t> upper;
    std::vector<uint32_t> lower;
    std::vector<uint32_t> first_leaf;
    std::vector<uint64_t> jump;
    std::vector<uint32_t> nbr;
    // device arena (one allocation) and the views into it
    void* arena = nullptr;
    size_t arena_bytes = 0;
    bool owns_arena = true;    // false: the arena is the caller's (vbm_build_device_noalloc)
    bool host_mirrors = true;  // false: no host copies of the arrays (vbm_build_device_noalloc)
    // Device-built grids fill the host arrays from the arena on first export.
    bool mirrors_filled = true;
    std::mutex mirror_mu;
    int device = -1;
    vbm::DevGrid dev{};
    // vbm_box_filter_batch_host: staging buffers and streams, made on first use
    std::mutex hostio_mu;
    vbm::HostIO* hostio = nullptr;
};

namespace vbm {

// Byte offsets of the grid's arrays in its one device allocation, in the order
// leaves, root_keys, upper, lower, first_leaf, jump, nbr, rowrank, rowrank_z
// (256-byte aligned).  The first seven have host copies; the row ranks are
// made on the device.
constexpr int kArenaArrays = 9, kHostArrays = 7;
struct ArenaLayout {
    size_t off[kArenaArrays];
    size_t bytes[kArenaArrays];
    size_t total;
};

inline ArenaLayout arena_layout(size_t n_leaves, size_t n_upper, size_t n_lower, size_t n_blocks, int log2w) {
    ArenaLayout a;
    const size_t words = ((size_t)1 << log2w) / 64;
    a.bytes[0] = n_leaves * sizeof(LeafRec);
    a.bytes[1] = n_upper * sizeof(uint64_t);
    a.bytes[2] = n_upper * (size_t)kUpperSlots * sizeof(uint32_t);
    a.bytes[3] = n_lower * (size_t)kLowerSlots * sizeof(uint32_t);
    a.bytes[4] = n_blocks * sizeof(uint32_t);
    a.bytes[5] = n_blocks * words * sizeof(uint64_t);
    a.bytes[6] = n_leaves * (size_t)kNbrStride * sizeof(uint32_t);
    a.bytes[7] = n_leaves * (size_t)kRowRanks * 2 * sizeof(uint32_t);
    a.bytes[8] = n_leaves * (size_t)kRowRanks * 4 * sizeof(uint32_t);
    size_t total = 0;
    for (int i = 0; i < kArenaArrays; ++i) {
        a.off[i] = total;
        total = (total + a.bytes[i] + 255) / 256 * 256;
    }
    a.total = total ? total : 256;
    return a;
}

// Device views of an arena laid out by arena_layout (sizes from g).
inline void set_device_views(vbm_grid* g, const ArenaLayout& a, int sm_count) {
    char* base = static_cast<char*>(g->arena);
    DevGrid& d = g->dev;
    d.leaves = reinterpret_cast<const LeafRec*>(base + a.off[0]);
    d.root_keys = reinterpret_cast<const uint64_t*>(base + a.off[1]);
    d.upper = reinterpret_cast<const uint32_t*>(base + a.off[2]);
    d.lower = reinterpret_cast<const uint32_t*>(base + a.off[3]);
    d.first_leaf = reinterpret_cast<const uint32_t*>(base + a.off[4]);
    d.jump = reinterpret_cast<const uint64_t*>(base + a.off[5]);
    d.nbr = reinterpret_cast<const uint32_t*>(base + a.off[6]);
    d.rowrank = reinterpret_cast<const uint2*>(base + a.off[7]);
    d.rowrank_z = reinterpret_cast<const uint4*>(base + a.off[8]);
    d.n = (uint32_t)g->n;
    d.n_leaves = (uint32_t)g->n_leaves;
    d.n_blocks = (uint32_t)g->n_blocks;
    d.n_upper = g->n_upper;
    d.log2w = g->log2w;
    d.sm_count = sm_count;
    d.block0 = 0;
}

// Host builder (vbm_build.cpp).  Fills every host array of g; returns a status
// code and sets err on failure.
int build_host(const int32_t* coords, uint64_t n, int log2w, uint32_t flags, vbm_grid* g, std::string& err);

// Device builder (vbm_build_dev.cu): coords is a device array of 3n int32.
// Fills the device arena and the host mirrors of g; synchronises `stream`.
int build_device(const int32_t* coords, uint64_t n, int log2w, uint32_t flags, void* stream, vbm_grid* g,
                 std::string& err);

// vbm_box_filter_batch_host (vbm_host.cu): arguments already checked; the
// grid's device is current.
int box_filter_batch_host(vbm_grid* g, int count, const float* const* host_sidecars, const int* C,
                          float* const* host_outs, int resolver, void* stream, std::string& err);

// Halo rows of the shard owning blocks [b0, b1) (vbm_shard.cu); the grid's
// host arrays must be filled.
void shard_halo(const vbm_grid* g, uint32_t b0, uint32_t b1, std::vector<uint32_t>& rows);

// Allocation-free device builder (vbm_build_device_noalloc): temporary memory
// in a static device array, the grid's arrays in the caller's `arena`.
int build_device_noalloc(const int32_t* coords, uint64_t n, int log2w, uint32_t flags, void* arena,
                         uint64_t arena_bytes, uint64_t* arena_needed, void* stream, vbm_grid* g, std::string& err);
}  // namespace vbm
