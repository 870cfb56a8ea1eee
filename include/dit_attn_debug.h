/*
 * dit_attn_debug.h -- extra entry points of the debug library,
 * libditattn_debug.so: the same sources as libditattn.so compiled with
 * DIT_DEBUG, exporting everything dit_attn.h declares plus the calls below.
 * The pages have no counterpart: this is test instrumentation for the
 * kernels' own failure handling and addressing.
 *
 * What the debug library adds to every attention call (dit_attn_fwd and its
 * _ws, _masked, _masked_noalloc, _accumulate and _fp8 forms):
 *   - In-kernel bounds checks.  The work item and key range a CTA decodes, the
 *     key tile of every K/V load, the shared-memory ring slots the products
 *     read, the mask words, and every O, LSE and workspace element written
 *     are checked against the extents the host derives from the arguments.
 *     A failed check records DIT_ERR_BOUNDS in the device status word (block,
 *     warp role, check site) and the access is skipped; the kernel carries on.
 *   - Fault injection (dit_debug_configure): one CTA withholds one producer
 *     signal, so that the warps waiting on it run into their bounded waits,
 *     report DIT_ERR_TIMEOUT and the whole CTA winds down -- the abort flag
 *     stops the other roles, copies and products already in flight are waited
 *     for (with a limit), tensor memory is released and the kernel returns.
 *     The context stays usable; the next call runs normally.
 * dit_check_watchdog() (dit_attn.h) reads and clears the report.
 *
 * The product library exports none of these calls and reports neither
 * condition: its kernels compile without the checks and the injection.
 */
#ifndef DIT_ATTN_DEBUG_H
#define DIT_ATTN_DEBUG_H

#include <stdint.h>

#include "dit_attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Kinds of injected fault. */
typedef enum {
    DIT_FAULT_NONE = 0,
    DIT_FAULT_SKIP_LOAD = 1,      /* the TMA thread skips K/V load `index` (K_j is
                                     load 2j, V_j load 2j+1 of the CTA's key
                                     tiles): no arrive, no copy               */
    DIT_FAULT_SKIP_S_COMMIT = 2,  /* the MMA warp skips the completion signal
                                     of S for query tile 0, key tile `index`  */
    DIT_FAULT_SKIP_P_ARRIVE = 3   /* softmax warp 0 (query tile 0) skips its
                                     "P ready" arrive at key tile `index`     */
} dit_debug_fault_t;

/*
 * dit_debug_configure -- settings every following attention call of this
 * process uses, until the next call of this function.
 * fault            a dit_debug_fault_t (DIT_FAULT_NONE: no injection).
 * fault_block      linear block index (x + gridX * (y + gridY * z)) of the CTA
 *                  that injects it, in every attention kernel the call
 *                  launches (use calls without a tail split to target one).
 * fault_index      which load / commit / arrive (see dit_debug_fault_t).
 * wait_limit_us    limit of every bounded in-kernel wait, 1,000 to 2,000,000
 *                  microseconds; 0 keeps the default (about two seconds).
 * out_extent_shrink  elements taken off the O extent the bounds checks
 *                  allow (0: the true extent).  A positive value makes the
 *                  stores to the last elements fail their check and be
 *                  skipped -- a way to see the checks fire without any access
 *                  outside the caller's buffer.
 * Returns DIT_ERR_INVALID_ARG for values outside these ranges.  Host only.
 */
dit_status_t dit_debug_configure(uint32_t fault, int fault_block, int fault_index, uint32_t wait_limit_us,
                                 int64_t out_extent_shrink);

/* 1 in the debug library (the symbol exists only there). */
uint32_t dit_debug_build(void);

#ifdef __cplusplus
}
#endif

#endif /* DIT_ATTN_DEBUG_H */
