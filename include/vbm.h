/*
 * vbm.h -- C ABI of libvbm.so, a GB300 (sm_103a) sparse voxel-grid stencil
 * library in the style of NanoVDB's VoxelBlockManager (VBM).
 *
 * Sources (web pages; cited by title and section):
 *   [2263] OpenVDB PR #2263 "Alternative stencil resolvers for VoxelBlockManager"
 *   [2262] OpenVDB PR #2262 "NanoVDB VBM: Streaming box-stencil"
 *   [2258] OpenVDB PR #2258 "VBM select-based inverse-map decode"
 *
 * Model.  An index grid ([2262] "What changed") maps each of N active voxels
 * to an index 1..N into a caller-owned sidecar; index 0 means background.  The
 * grid is a sparse tree of 8^3 leaves (512-bit value masks with a 9-bit
 * per-word prefix-sum directory, [2258] "Summary") under 16^3 lower and 32^3
 * upper nodes and a root table.  Indices are assigned in depth-first tree order:
 * upper nodes by signed (x>>12, y>>12, z>>12) lexicographically, then lower-node
 * slot, leaf slot and in-leaf offset off = (x&7)*64 + (y&7)*8 + (z&7), each slot
 * x-major.  The VBM cuts the index range into blocks of W = 2^log2 consecutive
 * indices (block b holds 1+b*W .. (b+1)*W); per block it stores firstLeafID
 * (leaf of the block's first index) and jumpMap (bit s, 1 <= s < W, set iff
 * index 1+b*W+s starts a leaf) ([2263] "Built on the register-decode API").
 *
 * Conventions for every call.
 *   - Return value: VBM_OK (0) or a negative VBM_ERR_* code; vbm_last_error()
 *     returns a text for the calling thread's last failure.  No call throws,
 *     traps or aborts.
 *   - Device pointers are caller-owned (e.g. torch allocations) and must point
 *     to memory on the device that was current when the grid was built; they
 *     must be 16-byte aligned.  A grid handle owns only its own arrays.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Compute
 *     calls only enqueue work: they return after launching, and launch errors
 *     are reported as VBM_ERR_CUDA.  Results are ready when the stream is.
 *     They allocate nothing and never synchronise, so they may be captured
 *     into a CUDA graph, and calls on one grid may run on several streams at
 *     once.  The builders allocate and synchronise (except
 *     vbm_build_device_noalloc after its first call on a device).
 *   - Sidecars and filter outputs hold (N+1) rows of C interleaved fp32
 *     channels: row r at [r*C, r*C+C).  Row 0 (background) is never read as a
 *     tap; filters write it as +0.0 so an output can serve as the next sidecar.
 *     Rows of a filter output are written only by that call: out must not
 *     overlap the sidecar (a shared byte is rejected with VBM_ERR_INVALID).
 *   - Limits: N < 2^31 (indices are 32-bit), |x|,|y|,|z| <= 2^30, C in 1..64,
 *     log2 block width in 6..9 (W = 64..512).
 */
#ifndef VBM_H
#define VBM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---- */
#define VBM_OK 0
#define VBM_ERR_INVALID (-1)   /* NULL pointer, unknown enum, C or log2 width out of range */
#define VBM_ERR_DUPLICATE (-2) /* a coordinate appears twice and VBM_BUILD_DEDUP was not given */
#define VBM_ERR_RANGE (-3)     /* N or a coordinate beyond the limits above */
#define VBM_ERR_NOMEM (-4)     /* host or device allocation failed */
#define VBM_ERR_CUDA (-5)      /* a CUDA runtime call or kernel launch failed */
#define VBM_ERR_ALIGN (-6)     /* a device pointer is not 16-byte aligned */
#define VBM_ERR_STATE (-7)     /* grid was built with VBM_BUILD_HOST_ONLY (no device arrays) */

/* MaxCachedLeaves: a block whose indices span more leaves than this resolves
 * its taps by tree walk instead of the cached table ([2263] "Notes":
 * MaxCachedLeaves is 16; "Summary": blocks spanning more fall back to per-tap
 * traversal). */
#define VBM_MAX_CACHED_LEAVES 16

/* vbm_build flags */
#define VBM_BUILD_DEDUP 1u     /* drop repeated coordinates instead of failing */
#define VBM_BUILD_HOST_ONLY 2u /* build the host arrays only (no CUDA calls); for inspection */

/* resolver: how a tap's index is found ([2263] "Summary" table) */
#define VBM_RESOLVE_TREEWALK 0 /* root-down tree traversal per tap; no shared memory */
#define VBM_RESOLVE_CACHED 1   /* per-block neighbour-leaf table staged in shared memory */
#define VBM_RESOLVE_BRICK 2    /* cached table + per-leaf padded index/value brick in shared memory
                                  (this library's GB300 resolver; no counterpart on the pages) */

/* output: how taps reach the consumer ([2262] "Summary", [2263] "Summary") */
#define VBM_OUTPUT_STREAMED 0     /* each (tap, index) consumed as it is resolved (forEach*) */
#define VBM_OUTPUT_MATERIALISED 1 /* all taps resolved into a per-thread array first (compute*) */

/* vbm_box_filter_batch: sidecars per call */
#define VBM_MAX_BATCH 8

/* cross-stencil consumer */
#define VBM_CROSS_LAPLACIAN 0 /* sum of the active face values (increasing tap order) - 6*centre */
#define VBM_CROSS_SUM 1       /* sum of the 7 taps' values in tap order */

/* vbm_leaf_export: which host array */
#define VBM_EXPORT_LEAF_MASK 0    /* n_leaves x 8 uint64: value masks, bit off%64 of word off/64 */
#define VBM_EXPORT_LEAF_PREFIX 1  /* n_leaves uint64: 9-bit field w-1 (w=1..7) = set bits in words 0..w-1 */
#define VBM_EXPORT_LEAF_FIRST 2   /* n_leaves uint32: index of the leaf's first active voxel */
#define VBM_EXPORT_LEAF_ORIGIN 3  /* n_leaves x 3 int32: leaf origin (multiple of 8) */
#define VBM_EXPORT_BLOCK_FIRST_LEAF 4 /* n_blocks uint32: firstLeafID */
#define VBM_EXPORT_BLOCK_JUMP 5   /* n_blocks x (W/64) uint64: jumpMap, bit s in word s/64 */
#define VBM_EXPORT_LEAF_NEIGHBOURS 6 /* n_leaves x 32 uint32: entry (dx+1)*9+(dy+1)*3+(dz+1) = id of the leaf
                                        at origin + 8*(dx,dy,dz) or 0xFFFFFFFF; entries 27..31 unused */

typedef struct vbm_grid vbm_grid;

typedef struct vbm_info_t {
    uint64_t n_active;            /* N */
    uint64_t n_leaves;
    uint64_t n_blocks;            /* ceil(N / W) */
    uint32_t block_width;         /* W */
    uint32_t log2_block_width;
    uint32_t n_upper;             /* 32^3 upper nodes */
    uint32_t n_lower;             /* 16^3 lower nodes */
    uint64_t n_blocks_over_cache; /* blocks spanning > VBM_MAX_CACHED_LEAVES leaves (tree-walk fallback) */
    uint32_t max_span;            /* most leaves any block spans (1 + popcount(jumpMap)) */
    uint32_t on_device;           /* 1 if device arrays exist */
    uint64_t device_bytes;        /* bytes of device memory the grid owns */
} vbm_info_t;

/* Text of the calling thread's last error ("" if none).  Valid until the
 * thread's next vbm_* call. */
const char* vbm_last_error(void);

/* Build the index grid and VBM block metadata from N active coordinates
 * (host array, coords[3*i .. 3*i+2] = x,y,z of voxel i, any order).  Uploads
 * the grid to the current device with copies on `stream` and synchronises the
 * stream before returning, so `coords` may be freed afterwards.  *out receives
 * a new handle (release with vbm_destroy).  N = 0 gives an empty grid.
 * Errors: INVALID (out NULL, coords NULL with n > 0, bad log2 width or flags),
 * RANGE, DUPLICATE, NOMEM, CUDA.  The index assignment and metadata follow
 * the model above ([2258] "Summary": the leaf mask, its 9-bit directory and
 * the block's jumpMap are what the decode reads). */
int vbm_build(const int32_t* coords, uint64_t n, int log2_block_width, uint32_t flags, void* stream,
              vbm_grid** out);

/* Build the same grid from coordinates already in device memory: coords is a
 * device array of 3n int32 on the current device (any order).  The work runs
 * on the GPU (leaf hash table, masks by atomic OR, a radix sort of the leaves
 * into tree order, scans for first indices and node ids, parallel fill of the
 * leaf records, child tables, VBM block metadata and neighbour rows); the
 * result equals vbm_build's array for array.  Temporary device memory is
 * allocated and freed inside the call: a leaf hash table of 12 bytes per slot,
 * first sized for one leaf per 16 voxels (about 1.5 bytes per voxel) and
 * rebuilt at 2n slots if the grid has more leaves, plus ~150 bytes per leaf.
 * It comes from a stream-ordered pool of the library's own per device that
 * keeps up to 2 GB between builds (the first build on a device creates it).
 * The call synchronises `stream`.  The grid lives on the device only; the
 * first vbm_leaf_export copies its arrays to the host (synchronously, once per
 * grid).  Requires
 * |x|,|y|,|z| < 2^20 (VBM_ERR_RANGE otherwise).  Errors: as vbm_build. */
int vbm_build_device(const int32_t* coords, uint64_t n, int log2_block_width, uint32_t flags, void* stream,
                     vbm_grid** out);

/* vbm_build_device without any device allocation.  No counterpart on the
 * pages: this is a library-level variant for callers that cannot call
 * cudaMalloc -- code inside an application whose device memory belongs to an
 * allocator it does not own, or code that runs while another host thread is
 * capturing work into a CUDA graph (cudaMalloc may synchronise the device and
 * is refused during a global-mode capture).  Such a caller passes, besides the
 * coordinates (device array of 3n int32), the output memory: `arena`, a
 * 256-byte aligned device buffer of `arena_bytes` bytes that receives the
 * grid's arrays.
 *   - Temporary memory is a file-scope static device array of about 9.2 MB,
 *     sized for at most 65,536 voxels; every GPU that loads libvbm.so holds it
 *     until the process exits.  Larger inputs fail with VBM_ERR_RANGE.
 *   - If `arena` is NULL or too small the call fails with VBM_ERR_RANGE; when
 *     `arena_needed` is not NULL it receives the bytes this grid needs (so a
 *     first call with arena_bytes = 0 is a size query).  Every grid needs at
 *     least 256 bytes, an empty one (n = 0) included.
 *   - The first call on each device looks up the static array's address
 *     (cudaGetSymbolAddress) with that device current; the lookup is
 *     thread-safe, and a failed lookup is retried by the next call.  Make that
 *     first call before any stream capture.
 *   - Every call uses the same static array, which keeps the previous call's
 *     contents (the call clears what must start empty).  Calls that overlap
 *     on the GPU -- on different streams or host threads -- race; serialise
 *     them.
 *   - The call reads small counts back to the host (cudaMemcpyAsync into host
 *     memory, then cudaStreamSynchronize) between its kernels.  While another
 *     thread captures a graph in cudaStreamCaptureModeGlobal, CUDA may refuse
 *     such calls from this thread; a capture that runs beside this call
 *     should use thread-local or relaxed mode.
 *   - The handle owns no device memory: vbm_destroy frees only the handle, and
 *     the caller frees `arena` after destroying it.  The handle keeps no host
 *     copies (vbm_leaf_export returns VBM_ERR_STATE); every compute call works
 *     on it as on any grid.
 * Requires |x|,|y|,|z| < 2^20.  Errors: INVALID, ALIGN, RANGE, DUPLICATE, CUDA. */
int vbm_build_device_noalloc(const int32_t* coords, uint64_t n, int log2_block_width, uint32_t flags, void* arena,
                             uint64_t arena_bytes, uint64_t* arena_needed, void* stream, vbm_grid** out);

/* Free a grid and its device arrays.  NULL is accepted.  The caller must make
 * sure no launched work still uses the grid (synchronise its streams first). */
int vbm_destroy(vbm_grid* grid);

/* Sizes and statistics of a grid.  Errors: INVALID. */
int vbm_info(const vbm_grid* grid, vbm_info_t* info);

/* Copy one of the grid's arrays (see VBM_EXPORT_*) into the host buffer dst,
 * which holds `bytes` bytes; the exact size is required.  For a grid built by
 * vbm_build_device the first call copies the arrays from the device (it
 * synchronises the device and may allocate host memory).  Errors: INVALID,
 * RANGE (bytes differs from the array's size), STATE (a
 * vbm_build_device_noalloc grid, which keeps no host copies), NOMEM, CUDA. */
int vbm_leaf_export(const vbm_grid* grid, int what, void* dst, uint64_t bytes);

/* Select-based inverse-map decode ([2258] "What changed"): for every slot of
 * every block, leaf_index[b*W+s] = firstLeafID[b] + popcount(jumpMap[b] bits
 * 0..s) and voxel_offset[b*W+s] = position of the r-th set bit of that leaf's
 * mask (r = index - the leaf's first index), found through the 9-bit prefix
 * directory and an in-word select.  Slots whose index 1+b*W+s exceeds N get
 * the sentinels leaf_index = 0xFFFFFFFF, voxel_offset = 0xFFFF ([2258]
 * "Validation").  Both outputs are device arrays of n_blocks*W entries.
 * Errors: INVALID, STATE, ALIGN, CUDA. */
int vbm_decode(const vbm_grid* grid, uint32_t* leaf_index, uint16_t* voxel_offset, void* stream);

/* Sweep decode, the design the select decode replaced ([2258] "What changed";
 * timed against it in [2258] "A/B — decode"): one CTA per block, whose threads
 * sweep all 512 voxel slots of every leaf overlapping the block and keep the
 * active voxels whose index lies in the block; O(span x 512) work per block.
 * Same arguments, outputs (bit for bit) and errors as vbm_decode.  Provided
 * to reproduce the select-versus-sweep comparison. */
int vbm_decode_sweep(const vbm_grid* grid, uint32_t* leaf_index, uint16_t* voxel_offset, void* stream);

/* 27-tap box filter ([2262] "What changed", "A/B"; [2263] "Measurements"): for
 * every active voxel v and channel ch,
 *     out[v*C+ch] = sum over taps t = (di+1)*9+(dj+1)*3+(dk+1), t = 0..26, of
 *                   sidecar[idx_t*C+ch] for each tap whose index idx_t != 0,
 * accumulated in fp32 from +0.0 in increasing t with round-to-nearest adds (no
 * reassociation), so every resolver/output combination gives the same bits.
 * Each slot is decoded in registers, its taps resolved by `resolver`
 * (VBM_RESOLVE_*) and consumed per `output` (VBM_OUTPUT_*); blocks spanning more
 * than VBM_MAX_CACHED_LEAVES leaves use the tree walk.  VBM_RESOLVE_BRICK
 * stages, for each leaf the block spans, a 10x10x10 brick of the leaf and its
 * one-voxel halo in shared memory (indices ranked once per brick row, then the
 * sidecar values), so each tap is one shared-memory read; it adds +0.0 for
 * inactive taps, which leaves an fp32 sum that started at +0.0 unchanged bit for
 * bit, so all resolvers agree.  `output` does not apply to it (must be
 * VBM_OUTPUT_STREAMED or VBM_OUTPUT_MATERIALISED; both run the same kernel).  sidecar and out are
 * device arrays of (N+1)*C floats.  Errors: INVALID, STATE, ALIGN, CUDA. */
int vbm_box_filter(const vbm_grid* grid, const float* sidecar, int C, float* out, int resolver, int output,
                   void* stream);

/* Several box filters on one grid in one call: out_i = the 27-tap box filter
 * of sidecars[i] with C[i] channels, for i < count (1..VBM_MAX_BATCH), each
 * exactly as vbm_box_filter(grid, sidecars[i], C[i], outs[i], resolver,
 * VBM_OUTPUT_STREAMED, stream) computes it.  With the brick resolver the
 * filters whose C is 1, 2, 3, 4, 8 or 16 run in launches of up to four, in
 * which each block is decoded and its index bricks built once for all of them
 * (and a C=1 and a C=3 filter read each tap's index once for both); other
 * widths and resolvers launch one filter after another.  The order of the
 * entries does not change any result.
 * sidecars, C and outs are host arrays of `count` entries; no output may
 * overlap a sidecar or another output (sidecars may overlap each other).
 * Errors: as vbm_box_filter, INVALID for a bad count or an overlap. */
int vbm_box_filter_batch(const vbm_grid* grid, int count, const float* const* sidecars, const int* C,
                         float* const* outs, int resolver, void* stream);

/* vbm_box_filter_batch on host-resident data: the end-to-end call for a
 * caller whose sidecars and outputs live in host memory.  host_sidecars[i] and
 * host_outs[i] are host arrays of (N+1)*C[i] floats (layout as on the device).
 * The call copies every sidecar to the device (one cudaMemcpyAsync each), runs
 * vbm_box_filter_batch on the device copies and copies every output back (one
 * cudaMemcpyAsync each); the results are bit for bit those of
 * vbm_box_filter_batch.  The copies and the filter run on the grid's own
 * streams, and `stream` waits for the last copy back: the outputs are ready,
 * and the host sidecars and outputs may be reused, once `stream` is
 * synchronised.  The call itself only enqueues.  The copies in are not
 * ordered after earlier work on `stream` (so that they overlap the previous
 * call's filter and copies back): the host sidecars are read as they are when
 * the copies run, and sidecars written by GPU work must be complete (that work
 * synchronised) before the call.
 *   - Device staging: the grid keeps two sets of device buffers (sidecars and
 *     outputs of one call each) and alternates between them, so that the
 *     copies of consecutive calls overlap the filter of the previous one.  A
 *     set is allocated, or grown, by the first call that needs it (that call
 *     allocates device memory and may wait for the set's previous use); calls
 *     whose batches fit allocate nothing.  vbm_destroy frees the sets.
 *   - Host memory: pinned memory (cudaHostAlloc, cudaHostRegister) gives
 *     asynchronous copies that overlap in both directions; pageable memory is
 *     accepted, and CUDA then copies synchronously with the calling thread.
 *   - Calls on one grid from several host threads are serialised by a lock.
 *   - Unlike the device-buffer compute calls, this call is not for stream
 *     capture: it may allocate, and it works on the grid's own streams.
 *   - No output may overlap a sidecar or another output (host byte ranges).
 * Errors: as vbm_box_filter_batch (INVALID for NULL host pointers), NOMEM
 * (staging allocation), CUDA. */
int vbm_box_filter_batch_host(const vbm_grid* grid, int count, const float* const* host_sidecars, const int* C,
                              float* const* host_outs, int resolver, void* stream);

/* ---- Block-range shards (one grid, several GPUs) ----
 * The path shards by VBM blocks: a block's voxels are consecutive indices and
 * span few consecutive leaves ([2263] "Summary"), so a contiguous range of
 * blocks owns a contiguous index range, and its box taps reach only the 27
 * neighbour leaves of its own leaves.  Every rank keeps the whole topology
 * (the grid), owns the sidecar rows of its index range, receives the rows of
 * its halo from their owners, and filters its own blocks.  No counterpart on
 * the pages (they run one GPU). */

/* Shard s of n_shards owns blocks block_begin[s] .. block_begin[s+1]-1;
 * block_begin (host, n_shards+1 entries) gets an even split of the blocks
 * (which holds the voxel counts within one block of equal: every block but the
 * last has W voxels).  Shard s then owns indices 1+block_begin[s]*W ..
 * min(N, block_begin[s+1]*W).  Errors: INVALID (NULL, n_shards < 1). */
int vbm_shard_blocks(const vbm_grid* grid, int n_shards, uint32_t* block_begin);

/* Halo of the shard that owns blocks [b0, b1): the sorted indices, outside
 * its own index range, of the active voxels of every leaf that is one of the
 * 27 neighbours of a leaf its blocks span -- a superset of the indices its box
 * (and cross) taps can reach.  Host computation from the grid's arrays (a
 * device-built grid copies them to the host on first use).  rows (host) has
 * room for `capacity` entries; *count receives the halo's size (a first call
 * with capacity 0 is a size query; VBM_ERR_RANGE if capacity is smaller).
 * Errors: INVALID (b0 >= b1 or b1 > n_blocks, NULL count), RANGE, STATE (a
 * grid without host copies), NOMEM. */
int vbm_shard_halo(const vbm_grid* grid, uint32_t b0, uint32_t b1, uint32_t* rows, uint64_t capacity,
                   uint64_t* count);

/* dst[k*C .. k*C+C) = src[rows[k]*C .. rows[k]*C+C) for k < count: the halo
 * rows another shard needs, packed for the exchange.  src and dst are device
 * arrays of floats, rows a device array of count uint32 (each < the rows of
 * src, not checked).  Errors: INVALID, ALIGN, CUDA. */
int vbm_gather_rows(const float* src, int C, const uint32_t* rows, uint64_t count, float* dst, void* stream);

/* dst[rows[k]*C .. +C) = src[k*C .. +C) for k < count: received halo rows
 * placed at their indices in the shard's sidecar (full (N+1)*C layout, only
 * the shard's own rows and its halo rows defined).  Errors: as
 * vbm_gather_rows. */
int vbm_scatter_rows(const float* src, int C, const uint32_t* rows, uint64_t count, float* dst, void* stream);

/* vbm_box_filter_batch restricted to the voxels of blocks [b0, b1): writes
 * only their output rows (and row 0 if b0 == 0); reads only sidecar rows of
 * those voxels and of their taps, i.e. the shard's own rows and its halo
 * (vbm_shard_halo).  Same results, bit for bit, as the whole-grid call on
 * those rows.  Errors: as vbm_box_filter_batch, INVALID for a bad range. */
int vbm_box_filter_batch_blocks(const vbm_grid* grid, uint32_t b0, uint32_t b1, int count,
                                const float* const* sidecars, const int* C, float* const* outs, int resolver,
                                void* stream);

/* 7-tap cross stencil (centre and the six face neighbours, taps t in
 * {4,10,12,13,14,16,22} of the box numbering) consumed as `op`:
 * VBM_CROSS_LAPLACIAN: out = s - 6*centre, s = +0.0 plus each active face
 * value in increasing t, the product and the difference rounded separately;
 * VBM_CROSS_SUM: the plain fp32 sum of the active taps' values in tap order.
 * Taps are materialised per thread, as in the pages' compute*CrossStencil*
 * ([2263] "Notes": there is no streaming cross resolver).  Errors as for
 * vbm_box_filter. */
int vbm_cross_filter(const vbm_grid* grid, const float* sidecar, int C, float* out, int resolver, int op,
                     void* stream);

/* 19-tap WENO consumer ([2258] "A/B - decode" names it beside the box and
 * the Laplacian; the pages give no formula, so this one is a reading): for
 * every active voxel v,
 *     out[v] = Godunov upwind squared gradient norm of the level set phi at v,
 * at unit spacing, from fifth-order WENO one-sided derivatives (Jiang & Shu
 * 1996; Jiang & Peng 2000; epsilon 1e-6).  Taps j = 0..18: the centre and the
 * voxels 1, 2, 3 steps away along each axis, in increasing (di,dj,dk)
 * lexicographic order; an inactive tap reads phi[0], the background value.
 * Per axis, with p[-3..3] the tap values and d[k] = p[k] - p[k-1]:
 *     minus = WENO5(d[-2], d[-1], d[0], d[1], d[2]),
 *     plus  = WENO5(d[3], d[2], d[1], d[0], d[-1]);
 * outside (phi[v] > iso) the axis term is max(max(minus,0)^2, min(plus,0)^2),
 * inside max(min(minus,0)^2, max(plus,0)^2); out[v] = x term + y term + z term
 * in that order.  All in fp32, each operation rounded separately (no FMA), so
 * every resolver gives the same bits.  Scale by 1/dx^2 for spacing dx.
 * phi and out: device arrays of N+1 floats (out may not overlap phi); out[0] is
 * written as +0.0.  resolver: VBM_RESOLVE_*.  Errors: INVALID, STATE, ALIGN,
 * CUDA. */
int vbm_weno_filter(const vbm_grid* grid, const float* phi, float iso, float* out, int resolver, void* stream);

/* Raw taps for byte-exact validation ([2263] "Validation": all taps of every
 * thread materialised to global memory): taps[v*27 + t] (box) or taps[v*7 + j]
 * (cross) is the index of that neighbour of voxel v, 0 if inactive; row 0 is
 * all zeros.  taps is a device array of (N+1)*27 or (N+1)*7 uint32.
 * Errors: INVALID, STATE, ALIGN, CUDA. */
int vbm_box_taps(const vbm_grid* grid, uint32_t* taps, int resolver, void* stream);
int vbm_cross_taps(const vbm_grid* grid, uint32_t* taps, int resolver, void* stream);

/* Raw taps of the 19-tap WENO stencil, as vbm_box_taps: taps[v*19 + j] is the
 * index of tap j of voxel v (order as in vbm_weno_filter), 0 if inactive; row
 * 0 is all zeros.  taps is a device array of (N+1)*19 uint32. */
int vbm_weno_taps(const vbm_grid* grid, uint32_t* taps, int resolver, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* VBM_H */
