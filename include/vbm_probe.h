/*
 * vbm_probe.h -- measurement probes of libvbm.so (C ABI).  No counterpart on
 * the pages: these calls compute nothing of the pipeline.  They launch kernels
 * with the launch shape of a grid's filters, so that a filter's time can be
 * set against the least time any kernel of that shape takes on the same GPU.
 *
 * Conventions as in vbm.h: status codes, `stream` a cudaStream_t, enqueue
 * only, no allocation, no synchronisation.
 */
#ifndef VBM_PROBE_H
#define VBM_PROBE_H

#include <stdint.h>

#include "vbm.h"

#ifdef __cplusplus
extern "C" {
#endif

/* What the probe kernel's CTAs do. */
#define VBM_PROBE_EMPTY 0    /* nothing: launch, CTA scheduling and retirement only */
#define VBM_PROBE_METADATA 1 /* each CTA loads its block's firstLeafID and jumpMap words (one dependent
                                DRAM round trip after an L2 flush) and stores nothing */
#define VBM_PROBE_CHAIN 2    /* each CTA follows the brick resolver's chain of dependent loads and
                                nothing else: block metadata -> the first spanned leaf's record ->
                                its neighbour row -> a neighbour leaf's mask word -> one sidecar
                                value (from `sidecar`) */

/* Launch one CTA per VBM block of `grid`, with the thread count and the
 * dynamic shared memory of the brick box filter at this block width (W
 * threads; the shared memory is reserved, not touched), doing `kind`
 * (VBM_PROBE_*).  `sidecar` (device, (N+1) floats) is read only by
 * VBM_PROBE_CHAIN and may be NULL otherwise.  Errors: INVALID (grid NULL,
 * unknown kind, sidecar NULL for VBM_PROBE_CHAIN), STATE, ALIGN, CUDA. */
int vbm_probe_launch(const vbm_grid* grid, int kind, const float* sidecar, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* VBM_PROBE_H */
