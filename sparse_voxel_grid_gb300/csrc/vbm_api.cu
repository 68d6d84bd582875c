// C ABI of libvbm.so (declared in include/vbm.h): argument checks, the grid's
// device arena, and dispatch to the kernel launchers.  Every entry point
// returns a status code; nothing throws across the boundary.
#include <cuda_runtime.h>

#include <cstring>
#include <vector>
#include <mutex>
#include <new>
#include <string>

#include "../../include/vbm_probe.h"
#include "vbm_internal.h"
#include "vbm_launch.h"

namespace {

thread_local std::string g_last_error;

int fail(int code, const std::string& msg) {
    g_last_error = msg;
    return code;
}

int fail_cuda(const char* what, cudaError_t e) {
    return fail(VBM_ERR_CUDA, std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")");
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Whether the byte ranges [a, a + abytes) and [b, b + bbytes) share a byte.
bool overlaps(const void* a, size_t abytes, const void* b, size_t bbytes) {
    const uintptr_t pa = (uintptr_t)a, pb = (uintptr_t)b;
    return abytes && bbytes && pa < pb + bbytes && pb < pa + abytes;
}

// Bytes of a sidecar or filter output of C channels: (N+1) rows.
size_t rows_bytes(const vbm_grid* g, int C) { return (size_t)(g->n + 1) * (size_t)C * sizeof(float); }

// Switches to the grid's device for the duration of a call.
class DeviceGuard {
   public:
    explicit DeviceGuard(int device) {
        if (cudaGetDevice(&prev_) != cudaSuccess) prev_ = -1;
        if (prev_ != device) ok_ = cudaSetDevice(device) == cudaSuccess; else prev_ = -1;
    }
    ~DeviceGuard() {
        if (prev_ >= 0) cudaSetDevice(prev_);
    }
    bool ok() const { return ok_; }

   private:
    int prev_ = -1;
    bool ok_ = true;
};

// Copies the host arrays into one device allocation and fills g->dev.
int upload(vbm_grid* g, cudaStream_t stream) {
    const vbm::ArenaLayout lay = vbm::arena_layout(g->leaves.size(), g->root_keys.size(), g->n_lower,
                                                   g->first_leaf.size(), g->log2w);
    const void* src[vbm::kHostArrays] = {g->leaves.data(), g->root_keys.data(), g->upper.data(), g->lower.data(),
                          g->first_leaf.data(), g->jump.data(), g->nbr.data()};
    cudaError_t e = cudaGetDevice(&g->device);
    if (e != cudaSuccess) return fail_cuda("vbm_build: cudaGetDevice", e);
    int sm_count = 0;
    e = cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, g->device);
    if (e != cudaSuccess) return fail_cuda("vbm_build: cudaDeviceGetAttribute", e);
    e = cudaMalloc(&g->arena, lay.total);
    if (e != cudaSuccess) {
        g->arena = nullptr;
        cudaGetLastError();
        return fail(VBM_ERR_NOMEM, std::string("vbm_build: cudaMalloc of ") + std::to_string(lay.total) +
                                       " bytes failed: " + cudaGetErrorString(e));
    }
    g->arena_bytes = lay.total;
    char* base = static_cast<char*>(g->arena);
    for (int i = 0; i < vbm::kHostArrays; ++i) {
        if (!lay.bytes[i]) continue;
        e = cudaMemcpyAsync(base + lay.off[i], src[i], lay.bytes[i], cudaMemcpyHostToDevice, stream);
        if (e != cudaSuccess) return fail_cuda("vbm_build: cudaMemcpyAsync", e);
    }
    e = vbm::launch_row_ranks(reinterpret_cast<const vbm::LeafRec*>(base + lay.off[0]),
                              reinterpret_cast<const uint32_t*>(base + lay.off[6]), (uint32_t)g->leaves.size(),
                              reinterpret_cast<uint2*>(base + lay.off[7]), reinterpret_cast<uint4*>(base + lay.off[8]),
                              stream);
    if (e != cudaSuccess) return fail_cuda("vbm_build: row ranks", e);
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return fail_cuda("vbm_build: cudaStreamSynchronize", e);
    vbm::set_device_views(g, lay, sm_count);
    e = vbm::prepare_device_kernels(g->device);
    if (e != cudaSuccess) return fail_cuda("vbm_build: kernel attributes", e);
    return VBM_OK;
}

// Host copies of a device-built grid's arrays, made on first use (the build
// itself keeps everything on the device).  Thread-safe; synchronous.
int fill_mirrors(const vbm_grid* cg) {
    vbm_grid* g = const_cast<vbm_grid*>(cg);
    std::lock_guard<std::mutex> lock(g->mirror_mu);
    if (g->mirrors_filled) return VBM_OK;
    const vbm::ArenaLayout lay = vbm::arena_layout(g->n_leaves, g->n_upper, g->n_lower, g->n_blocks, g->log2w);
    try {
        g->leaves.resize(g->n_leaves);
        g->root_keys.resize(g->n_upper);
        g->upper.resize((size_t)g->n_upper * vbm::kUpperSlots);
        g->lower.resize((size_t)g->n_lower * vbm::kLowerSlots);
        g->first_leaf.resize(g->n_blocks);
        g->jump.resize(g->n_blocks * ((1u << g->log2w) >> 6));
        g->nbr.resize((size_t)g->n_leaves * vbm::kNbrStride);
    } catch (const std::bad_alloc&) {
        return fail(VBM_ERR_NOMEM, "vbm_leaf_export: out of host memory");
    }
    void* dst[vbm::kHostArrays] = {g->leaves.data(), g->root_keys.data(), g->upper.data(), g->lower.data(),
                    g->first_leaf.data(), g->jump.data(), g->nbr.data()};
    DeviceGuard guard(g->device);
    if (!guard.ok()) return fail(VBM_ERR_CUDA, "vbm_leaf_export: cannot select the grid's device");
    const char* base = static_cast<const char*>(g->arena);
    for (int i = 0; i < vbm::kHostArrays; ++i) {
        if (!lay.bytes[i]) continue;
        const cudaError_t e = cudaMemcpy(dst[i], base + lay.off[i], lay.bytes[i], cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return fail_cuda("vbm_leaf_export: cudaMemcpy", e);
    }
    g->mirrors_filled = true;
    return VBM_OK;
}

// Common checks for the compute calls.
int check_grid(const vbm_grid* g, const char* fn) {
    if (!g) return fail(VBM_ERR_INVALID, std::string(fn) + ": grid is NULL");
    if (!g->arena) return fail(VBM_ERR_STATE, std::string(fn) + ": grid was built host-only (no device arrays)");
    return VBM_OK;
}

int check_ptr(const void* p, const char* fn, const char* name) {
    if (!p) return fail(VBM_ERR_INVALID, std::string(fn) + ": " + name + " is NULL");
    if (!aligned16(p)) return fail(VBM_ERR_ALIGN, std::string(fn) + ": " + name + " is not 16-byte aligned");
    return VBM_OK;
}

}  // namespace

extern "C" {

const char* vbm_last_error(void) { return g_last_error.c_str(); }

int vbm_build(const int32_t* coords, uint64_t n, int log2_block_width, uint32_t flags, void* stream,
              vbm_grid** out) {
    g_last_error.clear();
    if (!out) return fail(VBM_ERR_INVALID, "vbm_build: out is NULL");
    *out = nullptr;
    if (!coords && n) return fail(VBM_ERR_INVALID, "vbm_build: coords is NULL");
    if (log2_block_width < 6 || log2_block_width > 9)
        return fail(VBM_ERR_INVALID, "vbm_build: log2_block_width must be in 6..9");
    if (flags & ~(VBM_BUILD_DEDUP | VBM_BUILD_HOST_ONLY)) return fail(VBM_ERR_INVALID, "vbm_build: unknown flags");
    vbm_grid* g = new (std::nothrow) vbm_grid;
    if (!g) return fail(VBM_ERR_NOMEM, "vbm_build: out of host memory");
    int rc;
    try {
        std::string err;
        rc = vbm::build_host(coords, n, log2_block_width, flags, g, err);
        if (rc != VBM_OK) {
            delete g;
            return fail(rc, err);
        }
    } catch (const std::bad_alloc&) {
        delete g;
        return fail(VBM_ERR_NOMEM, "vbm_build: out of host memory");
    }
    if (!(flags & VBM_BUILD_HOST_ONLY)) {
        rc = upload(g, static_cast<cudaStream_t>(stream));
        if (rc != VBM_OK) {
            std::string msg = g_last_error;
            vbm_destroy(g);
            return fail(rc, msg);
        }
    }
    *out = g;
    return VBM_OK;
}

int vbm_build_device(const int32_t* coords, uint64_t n, int log2_block_width, uint32_t flags, void* stream,
                     vbm_grid** out) {
    g_last_error.clear();
    if (!out) return fail(VBM_ERR_INVALID, "vbm_build_device: out is NULL");
    *out = nullptr;
    if (!coords && n) return fail(VBM_ERR_INVALID, "vbm_build_device: coords is NULL");
    if (log2_block_width < 6 || log2_block_width > 9)
        return fail(VBM_ERR_INVALID, "vbm_build_device: log2_block_width must be in 6..9");
    if (flags & ~VBM_BUILD_DEDUP) return fail(VBM_ERR_INVALID, "vbm_build_device: unknown flags");
    vbm_grid* g = new (std::nothrow) vbm_grid;
    if (!g) return fail(VBM_ERR_NOMEM, "vbm_build_device: out of host memory");
    int rc;
    try {
        std::string err;
        rc = vbm::build_device(coords, n, log2_block_width, flags, stream, g, err);
        if (rc != VBM_OK) {
            vbm_destroy(g);
            return fail(rc, err);
        }
    } catch (const std::bad_alloc&) {
        vbm_destroy(g);
        return fail(VBM_ERR_NOMEM, "vbm_build_device: out of host memory");
    }
    *out = g;
    return VBM_OK;
}

int vbm_build_device_noalloc(const int32_t* coords, uint64_t n, int log2_block_width, uint32_t flags, void* arena,
                             uint64_t arena_bytes, uint64_t* arena_needed, void* stream, vbm_grid** out) {
    g_last_error.clear();
    if (arena_needed) *arena_needed = 0;
    if (!out) return fail(VBM_ERR_INVALID, "vbm_build_device_noalloc: out is NULL");
    *out = nullptr;
    if (!coords && n) return fail(VBM_ERR_INVALID, "vbm_build_device_noalloc: coords is NULL");
    if (log2_block_width < 6 || log2_block_width > 9)
        return fail(VBM_ERR_INVALID, "vbm_build_device_noalloc: log2_block_width must be in 6..9");
    if (flags & ~VBM_BUILD_DEDUP) return fail(VBM_ERR_INVALID, "vbm_build_device_noalloc: unknown flags");
    vbm_grid* g = new (std::nothrow) vbm_grid;
    if (!g) return fail(VBM_ERR_NOMEM, "vbm_build_device_noalloc: out of host memory");
    std::string err;
    const int rc = vbm::build_device_noalloc(coords, n, log2_block_width, flags, arena, arena_bytes, arena_needed,
                                             stream, g, err);
    if (rc != VBM_OK) {
        delete g;  // owns no device memory
        return fail(rc, err);
    }
    *out = g;
    return VBM_OK;
}

int vbm_destroy(vbm_grid* g) {
    g_last_error.clear();
    if (!g) return VBM_OK;
    int rc = VBM_OK;
    if (g->hostio || (g->arena && g->owns_arena)) {  // host-only grids make no CUDA call
        DeviceGuard guard(g->device);
        if (g->hostio) {
            vbm::destroy_host_io(g->hostio);
            g->hostio = nullptr;
        }
        if (g->arena && g->owns_arena) {
            cudaError_t e = cudaFree(g->arena);
            if (e != cudaSuccess) rc = fail_cuda("vbm_destroy: cudaFree", e);
        }
    }
    delete g;
    return rc;
}

int vbm_info(const vbm_grid* g, vbm_info_t* info) {
    g_last_error.clear();
    if (!g || !info) return fail(VBM_ERR_INVALID, "vbm_info: NULL argument");
    std::memset(info, 0, sizeof(*info));
    info->n_active = g->n;
    info->n_leaves = g->n_leaves;
    info->n_blocks = g->n_blocks;
    info->block_width = 1u << g->log2w;
    info->log2_block_width = (uint32_t)g->log2w;
    info->n_upper = g->n_upper;
    info->n_lower = g->n_lower;
    info->n_blocks_over_cache = g->n_over_cache;
    info->max_span = g->max_span;
    info->on_device = g->arena ? 1u : 0u;
    info->device_bytes = g->arena_bytes;
    return VBM_OK;
}

int vbm_leaf_export(const vbm_grid* g, int what, void* dst, uint64_t bytes) {
    g_last_error.clear();
    if (!g || (!dst && bytes)) return fail(VBM_ERR_INVALID, "vbm_leaf_export: NULL argument");
    if (!g->host_mirrors) return fail(VBM_ERR_STATE, "vbm_leaf_export: this grid keeps no host copies");
    if (int rc = fill_mirrors(g)) return rc;
    const size_t nl = g->leaves.size();
    size_t need = 0;
    switch (what) {
        case VBM_EXPORT_LEAF_MASK: need = nl * 8 * sizeof(uint64_t); break;
        case VBM_EXPORT_LEAF_PREFIX: need = nl * sizeof(uint64_t); break;
        case VBM_EXPORT_LEAF_FIRST: need = nl * sizeof(uint32_t); break;
        case VBM_EXPORT_LEAF_ORIGIN: need = nl * 3 * sizeof(int32_t); break;
        case VBM_EXPORT_BLOCK_FIRST_LEAF: need = g->first_leaf.size() * sizeof(uint32_t); break;
        case VBM_EXPORT_BLOCK_JUMP: need = g->jump.size() * sizeof(uint64_t); break;
        case VBM_EXPORT_LEAF_NEIGHBOURS: need = g->nbr.size() * sizeof(uint32_t); break;
        default: return fail(VBM_ERR_INVALID, "vbm_leaf_export: unknown array");
    }
    if (bytes != need)
        return fail(VBM_ERR_RANGE, "vbm_leaf_export: expected " + std::to_string(need) + " bytes, got " +
                                       std::to_string(bytes));
    char* out = static_cast<char*>(dst);
    for (size_t l = 0; l < nl; ++l) {
        const vbm::LeafRec& r = g->leaves[l];
        switch (what) {
            case VBM_EXPORT_LEAF_MASK: std::memcpy(out + l * 64, r.mask, 64); break;
            case VBM_EXPORT_LEAF_PREFIX: std::memcpy(out + l * 8, &r.prefix, 8); break;
            case VBM_EXPORT_LEAF_FIRST: std::memcpy(out + l * 4, &r.first, 4); break;
            case VBM_EXPORT_LEAF_ORIGIN: std::memcpy(out + l * 12, r.origin, 12); break;
            default: break;
        }
    }
    if (what == VBM_EXPORT_BLOCK_FIRST_LEAF && need) std::memcpy(out, g->first_leaf.data(), need);
    if (what == VBM_EXPORT_BLOCK_JUMP && need) std::memcpy(out, g->jump.data(), need);
    if (what == VBM_EXPORT_LEAF_NEIGHBOURS && need) std::memcpy(out, g->nbr.data(), need);
    return VBM_OK;
}

int vbm_decode(const vbm_grid* g, uint32_t* leaf_index, uint16_t* voxel_offset, void* stream) {
    g_last_error.clear();
    int rc = check_grid(g, "vbm_decode");
    if (rc) return rc;
    if (g->n_blocks == 0) return VBM_OK;
    if ((rc = check_ptr(leaf_index, "vbm_decode", "leaf_index"))) return rc;
    if ((rc = check_ptr(voxel_offset, "vbm_decode", "voxel_offset"))) return rc;
    DeviceGuard guard(g->device);
    if (!guard.ok()) return fail(VBM_ERR_CUDA, "vbm_decode: cannot select the grid's device");
    cudaError_t e = vbm::launch_decode(g->dev, leaf_index, voxel_offset, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? VBM_OK : fail_cuda("vbm_decode: launch", e);
}

int vbm_decode_sweep(const vbm_grid* g, uint32_t* leaf_index, uint16_t* voxel_offset, void* stream) {
    g_last_error.clear();
    int rc = check_grid(g, "vbm_decode_sweep");
    if (rc) return rc;
    if (g->n_blocks == 0) return VBM_OK;
    if ((rc = check_ptr(leaf_index, "vbm_decode_sweep", "leaf_index"))) return rc;
    if ((rc = check_ptr(voxel_offset, "vbm_decode_sweep", "voxel_offset"))) return rc;
    DeviceGuard guard(g->device);
    if (!guard.ok()) return fail(VBM_ERR_CUDA, "vbm_decode_sweep: cannot select the grid's device");
    cudaError_t e = vbm::launch_sweep_decode(g->dev, leaf_index, voxel_offset, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? VBM_OK : fail_cuda("vbm_decode_sweep: launch", e);
}

static int check_filter(const vbm_grid* g, const float* sidecar, int C, const float* out, int resolver,
                        const char* fn) {
    int rc = check_grid(g, fn);
    if (rc) return rc;
    if (C < 1 || C > vbm::kMaxC) return fail(VBM_ERR_INVALID, std::string(fn) + ": C must be in 1..64");
    if (resolver != VBM_RESOLVE_TREEWALK && resolver != VBM_RESOLVE_CACHED && resolver != VBM_RESOLVE_BRICK)
        return fail(VBM_ERR_INVALID, std::string(fn) + ": unknown resolver");
    if ((rc = check_ptr(sidecar, fn, "sidecar"))) return rc;
    if ((rc = check_ptr(out, fn, "out"))) return rc;
    if (overlaps(sidecar, rows_bytes(g, C), out, rows_bytes(g, C)))
        return fail(VBM_ERR_INVALID, std::string(fn) + ": out overlaps sidecar");
    return VBM_OK;
}

int vbm_box_filter(const vbm_grid* g, const float* sidecar, int C, float* out, int resolver, int output,
                   void* stream) {
    g_last_error.clear();
    int rc = check_filter(g, sidecar, C, out, resolver, "vbm_box_filter");
    if (rc) return rc;
    if (output != VBM_OUTPUT_STREAMED && output != VBM_OUTPUT_MATERIALISED)
        return fail(VBM_ERR_INVALID, "vbm_box_filter: unknown output mode");
    DeviceGuard guard(g->device);
    if (!guard.ok()) return fail(VBM_ERR_CUDA, "vbm_box_filter: cannot select the grid's device");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (g->n_blocks == 0) e = cudaMemsetAsync(out, 0, sizeof(float) * (size_t)C, s);
    else if (resolver == VBM_RESOLVE_BRICK) e = vbm::launch_brick_box(g->dev, sidecar, C, out, s);
    else e = vbm::launch_box_filter(g->dev, sidecar, C, out, resolver, output, s);
    return e == cudaSuccess ? VBM_OK : fail_cuda("vbm_box_filter: launch", e);
}

int vbm_box_filter_batch(const vbm_grid* g, int count, const float* const* sidecars, const int* C,
                         float* const* outs, int resolver, void* stream) {
    g_last_error.clear();
    const char* fn = "vbm_box_filter_batch";
    if (count < 1 || count > VBM_MAX_BATCH) return fail(VBM_ERR_INVALID, std::string(fn) + ": count must be in 1..8");
    if (!sidecars || !C || !outs) return fail(VBM_ERR_INVALID, std::string(fn) + ": NULL array");
    for (int i = 0; i < count; ++i) {
        int rc = check_filter(g, sidecars[i], C[i], outs[i], resolver, fn);
        if (rc) return rc;
        for (int j = 0; j < i; ++j) {
            if (overlaps(outs[i], rows_bytes(g, C[i]), sidecars[j], rows_bytes(g, C[j])) ||
                overlaps(outs[j], rows_bytes(g, C[j]), sidecars[i], rows_bytes(g, C[i])))
                return fail(VBM_ERR_INVALID, std::string(fn) + ": an output overlaps a sidecar");
            if (overlaps(outs[i], rows_bytes(g, C[i]), outs[j], rows_bytes(g, C[j])))
                return fail(VBM_ERR_INVALID, std::string(fn) + ": two outputs overlap");
        }
    }
    DeviceGuard guard(g->device);
    if (!guard.ok()) return fail(VBM_ERR_CUDA, std::string(fn) + ": cannot select the grid's device");
    const cudaError_t e = vbm::launch_box_batch(g->dev, count, sidecars, C, outs, resolver,
                                                static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? VBM_OK : fail_cuda("vbm_box_filter_batch: launch", e);
}

int vbm_box_filter_batch_host(const vbm_grid* cg, int count, const float* const* host_sidecars, const int* C,
                              float* const* host_outs, int resolver, void* stream) {
    g_last_error.clear();
    const char* fn = "vbm_box_filter_batch_host";
    int rc = check_grid(cg, fn);
    if (rc) return rc;
    if (count < 1 || count > VBM_MAX_BATCH) return fail(VBM_ERR_INVALID, std::string(fn) + ": count must be in 1..8");
    if (!host_sidecars || !C || !host_outs) return fail(VBM_ERR_INVALID, std::string(fn) + ": NULL array");
    if (resolver != VBM_RESOLVE_TREEWALK && resolver != VBM_RESOLVE_CACHED && resolver != VBM_RESOLVE_BRICK)
        return fail(VBM_ERR_INVALID, std::string(fn) + ": unknown resolver");
    for (int i = 0; i < count; ++i) {
        if (C[i] < 1 || C[i] > vbm::kMaxC) return fail(VBM_ERR_INVALID, std::string(fn) + ": C must be in 1..64");
        if (!host_sidecars[i] || !host_outs[i])
            return fail(VBM_ERR_INVALID, std::string(fn) + ": a host sidecar or output is NULL");
        for (int j = 0; j <= i; ++j) {
            if (overlaps(host_outs[i], rows_bytes(cg, C[i]), host_sidecars[j], rows_bytes(cg, C[j])) ||
                overlaps(host_outs[j], rows_bytes(cg, C[j]), host_sidecars[i], rows_bytes(cg, C[i])))
                return fail(VBM_ERR_INVALID, std::string(fn) + ": an output overlaps a sidecar");
            if (j < i && overlaps(host_outs[i], rows_bytes(cg, C[i]), host_outs[j], rows_bytes(cg, C[j])))
                return fail(VBM_ERR_INVALID, std::string(fn) + ": two outputs overlap");
        }
    }
    DeviceGuard guard(cg->device);
    if (!guard.ok()) return fail(VBM_ERR_CUDA, std::string(fn) + ": cannot select the grid's device");
    std::string err;
    rc = vbm::box_filter_batch_host(const_cast<vbm_grid*>(cg), count, host_sidecars, C, host_outs, resolver, stream,
                                    err);
    return rc == VBM_OK ? VBM_OK : fail(rc, err);
}

int vbm_shard_blocks(const vbm_grid* g, int n_shards, uint32_t* block_begin) {
    g_last_error.clear();
    if (!g || !block_begin) return fail(VBM_ERR_INVALID, "vbm_shard_blocks: NULL argument");
    if (n_shards < 1) return fail(VBM_ERR_INVALID, "vbm_shard_blocks: n_shards must be at least 1");
    for (int s = 0; s <= n_shards; ++s) block_begin[s] = (uint32_t)(g->n_blocks * (uint64_t)s / (uint64_t)n_shards);
    return VBM_OK;
}

int vbm_shard_halo(const vbm_grid* g, uint32_t b0, uint32_t b1, uint32_t* rows, uint64_t capacity,
                   uint64_t* count) {
    g_last_error.clear();
    const char* fn = "vbm_shard_halo";
    if (!g || !count) return fail(VBM_ERR_INVALID, std::string(fn) + ": NULL argument");
    *count = 0;
    if (b0 > b1 || b1 > g->n_blocks) return fail(VBM_ERR_INVALID, std::string(fn) + ": bad block range");
    if (!g->host_mirrors) return fail(VBM_ERR_STATE, std::string(fn) + ": this grid keeps no host copies");
    if (int rc = fill_mirrors(g)) return rc;
    std::vector<uint32_t> halo;
    try {
        vbm::shard_halo(g, b0, b1, halo);
    } catch (const std::bad_alloc&) {
        return fail(VBM_ERR_NOMEM, std::string(fn) + ": out of host memory");
    }
    *count = halo.size();
    if (capacity < halo.size()) {
        if (capacity == 0 && !rows) return VBM_OK;  // size query
        return fail(VBM_ERR_RANGE, std::string(fn) + ": rows holds " + std::to_string(capacity) + " entries; the halo has " +
                                       std::to_string(halo.size()));
    }
    if (!halo.empty()) {
        if (!rows) return fail(VBM_ERR_INVALID, std::string(fn) + ": rows is NULL");
        std::memcpy(rows, halo.data(), halo.size() * sizeof(uint32_t));
    }
    return VBM_OK;
}

static int rows_call(bool gather, const float* src, int C, const uint32_t* rows, uint64_t count, float* dst,
                     void* stream) {
    const char* fn = gather ? "vbm_gather_rows" : "vbm_scatter_rows";
    if (C < 1 || C > vbm::kMaxC) return fail(VBM_ERR_INVALID, std::string(fn) + ": C must be in 1..64");
    if (count == 0) return VBM_OK;
    int rc;
    if ((rc = check_ptr(src, fn, "src")) || (rc = check_ptr(rows, fn, "rows")) || (rc = check_ptr(dst, fn, "dst")))
        return rc;
    const cudaError_t e = vbm::launch_rows(gather, src, C, rows, count, dst, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? VBM_OK : fail_cuda((std::string(fn) + ": launch").c_str(), e);
}

int vbm_gather_rows(const float* src, int C, const uint32_t* rows, uint64_t count, float* dst, void* stream) {
    g_last_error.clear();
    return rows_call(true, src, C, rows, count, dst, stream);
}

int vbm_scatter_rows(const float* src, int C, const uint32_t* rows, uint64_t count, float* dst, void* stream) {
    g_last_error.clear();
    return rows_call(false, src, C, rows, count, dst, stream);
}

int vbm_box_filter_batch_blocks(const vbm_grid* g, uint32_t b0, uint32_t b1, int count,
                                const float* const* sidecars, const int* C, float* const* outs, int resolver,
                                void* stream) {
    g_last_error.clear();
    const char* fn = "vbm_box_filter_batch_blocks";
    int rc = check_grid(g, fn);
    if (rc) return rc;
    if (b0 > b1 || b1 > g->n_blocks) return fail(VBM_ERR_INVALID, std::string(fn) + ": bad block range");
    if (count < 1 || count > VBM_MAX_BATCH) return fail(VBM_ERR_INVALID, std::string(fn) + ": count must be in 1..8");
    if (!sidecars || !C || !outs) return fail(VBM_ERR_INVALID, std::string(fn) + ": NULL array");
    for (int i = 0; i < count; ++i) {
        if ((rc = check_filter(g, sidecars[i], C[i], outs[i], resolver, fn))) return rc;
        for (int j = 0; j < i; ++j) {
            if (overlaps(outs[i], rows_bytes(g, C[i]), sidecars[j], rows_bytes(g, C[j])) ||
                overlaps(outs[j], rows_bytes(g, C[j]), sidecars[i], rows_bytes(g, C[i])))
                return fail(VBM_ERR_INVALID, std::string(fn) + ": an output overlaps a sidecar");
            if (overlaps(outs[i], rows_bytes(g, C[i]), outs[j], rows_bytes(g, C[j])))
                return fail(VBM_ERR_INVALID, std::string(fn) + ": two outputs overlap");
        }
    }
    if (b0 == b1) return VBM_OK;
    DeviceGuard guard(g->device);
    if (!guard.ok()) return fail(VBM_ERR_CUDA, std::string(fn) + ": cannot select the grid's device");
    vbm::DevGrid view = g->dev;
    view.block0 = b0;
    view.n_blocks = b1 - b0;
    const cudaError_t e = vbm::launch_box_batch(view, count, sidecars, C, outs, resolver, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? VBM_OK : fail_cuda("vbm_box_filter_batch_blocks: launch", e);
}

int vbm_cross_filter(const vbm_grid* g, const float* sidecar, int C, float* out, int resolver, int op,
                     void* stream) {
    g_last_error.clear();
    int rc = check_filter(g, sidecar, C, out, resolver, "vbm_cross_filter");
    if (rc) return rc;
    if (op != VBM_CROSS_LAPLACIAN && op != VBM_CROSS_SUM)
        return fail(VBM_ERR_INVALID, "vbm_cross_filter: unknown op");
    DeviceGuard guard(g->device);
    if (!guard.ok()) return fail(VBM_ERR_CUDA, "vbm_cross_filter: cannot select the grid's device");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (g->n_blocks == 0) e = cudaMemsetAsync(out, 0, sizeof(float) * (size_t)C, s);
    else if (resolver == VBM_RESOLVE_BRICK) e = vbm::launch_brick_cross(g->dev, sidecar, C, out, op, s);
    else e = vbm::launch_cross_filter(g->dev, sidecar, C, out, resolver, op, s);
    return e == cudaSuccess ? VBM_OK : fail_cuda("vbm_cross_filter: launch", e);
}

static int taps_common(const vbm_grid* g, uint32_t* taps, int resolver, void* stream, bool box) {
    const char* fn = box ? "vbm_box_taps" : "vbm_cross_taps";
    int rc = check_grid(g, fn);
    if (rc) return rc;
    if (resolver != VBM_RESOLVE_TREEWALK && resolver != VBM_RESOLVE_CACHED && resolver != VBM_RESOLVE_BRICK)
        return fail(VBM_ERR_INVALID, std::string(fn) + ": unknown resolver");
    if ((rc = check_ptr(taps, fn, "taps"))) return rc;
    DeviceGuard guard(g->device);
    if (!guard.ok()) return fail(VBM_ERR_CUDA, std::string(fn) + ": cannot select the grid's device");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (g->n_blocks == 0) e = cudaMemsetAsync(taps, 0, sizeof(uint32_t) * (box ? vbm::kBoxTaps : vbm::kCrossTaps), s);
    else if (resolver == VBM_RESOLVE_BRICK) e = vbm::launch_brick_taps(g->dev, taps, box ? vbm::kBoxTaps : vbm::kCrossTaps, s);
    else e = box ? vbm::launch_box_taps(g->dev, taps, resolver, s) : vbm::launch_cross_taps(g->dev, taps, resolver, s);
    return e == cudaSuccess ? VBM_OK : fail_cuda((std::string(fn) + ": launch").c_str(), e);
}

int vbm_weno_filter(const vbm_grid* g, const float* phi, float iso, float* out, int resolver, void* stream) {
    g_last_error.clear();
    int rc = check_filter(g, phi, 1, out, resolver, "vbm_weno_filter");
    if (rc) return rc;
    DeviceGuard guard(g->device);
    if (!guard.ok()) return fail(VBM_ERR_CUDA, "vbm_weno_filter: cannot select the grid's device");
    cudaError_t e = vbm::launch_weno_filter(g->dev, phi, iso, out, resolver, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? VBM_OK : fail_cuda("vbm_weno_filter: launch", e);
}

int vbm_weno_taps(const vbm_grid* g, uint32_t* taps, int resolver, void* stream) {
    g_last_error.clear();
    int rc = check_grid(g, "vbm_weno_taps");
    if (rc) return rc;
    if (resolver != VBM_RESOLVE_TREEWALK && resolver != VBM_RESOLVE_CACHED && resolver != VBM_RESOLVE_BRICK)
        return fail(VBM_ERR_INVALID, "vbm_weno_taps: unknown resolver");
    if ((rc = check_ptr(taps, "vbm_weno_taps", "taps"))) return rc;
    DeviceGuard guard(g->device);
    if (!guard.ok()) return fail(VBM_ERR_CUDA, "vbm_weno_taps: cannot select the grid's device");
    cudaError_t e = vbm::launch_weno_taps(g->dev, taps, resolver, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? VBM_OK : fail_cuda("vbm_weno_taps: launch", e);
}

int vbm_box_taps(const vbm_grid* g, uint32_t* taps, int resolver, void* stream) {
    g_last_error.clear();
    return taps_common(g, taps, resolver, stream, true);
}

int vbm_cross_taps(const vbm_grid* g, uint32_t* taps, int resolver, void* stream) {
    g_last_error.clear();
    return taps_common(g, taps, resolver, stream, false);
}

int vbm_probe_launch(const vbm_grid* g, int kind, const float* sidecar, void* stream) {
    g_last_error.clear();
    const char* fn = "vbm_probe_launch";
    int rc = check_grid(g, fn);
    if (rc) return rc;
    if (kind != VBM_PROBE_EMPTY && kind != VBM_PROBE_METADATA && kind != VBM_PROBE_CHAIN)
        return fail(VBM_ERR_INVALID, std::string(fn) + ": unknown kind");
    if (kind == VBM_PROBE_CHAIN && (rc = check_ptr(sidecar, fn, "sidecar"))) return rc;
    if (g->n_blocks == 0) return VBM_OK;
    DeviceGuard guard(g->device);
    if (!guard.ok()) return fail(VBM_ERR_CUDA, std::string(fn) + ": cannot select the grid's device");
    const cudaError_t e = vbm::launch_probe(g->dev, kind, sidecar, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? VBM_OK : fail_cuda("vbm_probe_launch: launch", e);
}

}  // extern "C"
