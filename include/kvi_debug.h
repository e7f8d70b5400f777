/*
 * kvi_debug.h -- checks and failure hooks of the debug build of libkvi.
 *
 * The debug build is the same library compiled with -DKVI_DEBUG_CHECKS
 * (pre_rope_kv_gb300/build.py: build(debug=True) writes
 * pre_rope_kv_gb300/_build/libkvi_debug.so).  It differs from the release
 * build in two ways:
 *
 *   - kvi_inject_paged / kvi_inject_paged_ex first check, on the device, that
 *     no two injected facts' target ranges [start, start + fact_len) overlap
 *     (Section 5.1 places every fact at positions of its own; two facts
 *     written over the same slots are caller error).  An overlap is recorded
 *     as KVI_ERR_INVALID_ARG in *d_status; the injection still runs and its
 *     result on the overlapping slots is unspecified, as in the release
 *     build, which does not check.
 *   - it exports the hooks below, which let a test make one of the scoring
 *     kernels' bounded waits run out without a fault.
 *
 * Only the debug library exports the symbols declared here.
 */
#ifndef KVI_DEBUG_H
#define KVI_DEBUG_H

#include "kvi.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Failure hook (debug build only).  From the next call on, the scoring
 * kernel of the exact scan (kvi_retrieve_topk, kvi_retrieve_and_inject*)
 * stages no copy for the fact at flat row `row` of its R x max_facts row
 * space (row = request * max_facts + fact id), so that the consumer waiting
 * for it gives up after the kernel's one-second bound: the call's status
 * word then reads KVI_ERR_TIMEOUT and its outputs are not valid.  The waits
 * that depend on the missing row give up the same way, each after its
 * bound, and every copy the kernel did issue is waited for before it exits:
 * nothing faults and the context stays usable.  row < 0 turns the hook off.
 * Synchronous (it writes a device variable of the current device).
 * Errors: KVI_ERR_CUDA. */
KVI_API kvi_status kvi_debug_stall_scorer_row(int64_t row);

/* Failure hook (debug build only).  From the next call on, the tensor-core
 * kernel of the shared-store path (kvi_retrieve_topk_shared,
 * kvi_retrieve_and_inject_shared, the graph build) loads nothing for K chunk
 * `chunk` (32 floats of E) in its CTA `cta`: the waits on that stage give up
 * after the kernel's one-second bound, the call's status word reads
 * KVI_ERR_TIMEOUT and its outputs are not valid.  Every copy the CTA did
 * issue is waited for before it exits, and every CTA of a thread-block
 * cluster still reaches the cluster's barriers: nothing faults or hangs and
 * the context stays usable.  A (cta, chunk) that the launch does not have
 * changes nothing; cta < 0 turns the hook off.  Synchronous (it writes
 * device variables of the current device).  Errors: KVI_ERR_CUDA. */
KVI_API kvi_status kvi_debug_stall_coarse_chunk(int32_t cta, int32_t chunk);

#ifdef __cplusplus
}
#endif

#endif /* KVI_DEBUG_H */
