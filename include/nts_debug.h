/*
 * nts_debug.h -- tuning overrides and test hooks of libnts.  Not needed by
 * normal callers.  Settings are process-wide and apply to every later call
 * until changed; they are not thread-safe with respect to calls in flight on
 * other host threads.  No source page defines these: they exist to sweep
 * launch shapes and to exercise the library's error paths without faulting a
 * GPU.
 */
#ifndef NTS_DEBUG_H
#define NTS_DEBUG_H

#include <stdint.h>

#include "nts.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Override the automatic launch shape.  Each argument 0 means automatic.
 *   vpt        QK kernel: 16-byte vectors per thread, one of {1,2,3,4,5,6,8};
 *              MX kernels: MX blocks per thread (halves of 64-value
 *              blocks for B = 64), 1..8 with at most 16 vectors per thread
 *   rows       token rows per tile (rows * threads-per-row <= 480)
 *   stages     shared-memory ring stages (>= 1)
 *   grid       CTAs (MX kernels) or clusters (QK kernel) of the persistent grid
 *   smem_budget bytes a CTA's ring aims to stay under (default 102400)
 * Errors: INVALID_ARG for negative values or vpt > 8.  A shape the
 * device cannot run is reported by the next call as UNSUPPORTED or CUDA.
 */
NTS_API int nts_debug_set_tuning(int vpt, int rows, int stages, int64_t grid, int smem_budget);

/* Limit of every bounded in-kernel wait, in ns (0 = default, 1 s). */
NTS_API int nts_debug_set_wait_limit_ns(uint64_t ns);

/*
 * Tile order of the persistent kernels: 1 (default) = every CTA takes its next
 * tile from a per-stream counter; 0 = a fixed round-robin order.  Results do
 * not depend on it.  Errors: INVALID_ARG for other values.
 */
NTS_API int nts_debug_set_schedule(int dynamic);

/*
 * Decode-sized QK-RMSNorm and LayerNorm launches (bf16 output, every tile
 * in one wave of single-tile clusters, no launch-shape override and no
 * missing-bytes hook): 1 (default) = the
 * single-tile kernel without producer warp or ring; 0 = the persistent
 * kernel.  Results are identical either way.  Errors: INVALID_ARG for other
 * values.
 */
NTS_API int nts_debug_set_direct(int on);

/*
 * Chunking of the host-buffer forms: a call moves its rows in at most
 * max_chunks chunks (1..64) of at least min_chunk_bytes of input each; 0
 * restores a default (16 chunks, 16 MiB).  Results do not depend on it.
 * Errors: INVALID_ARG for values out of range.
 */
NTS_API int nts_debug_set_host_chunks(int max_chunks, int64_t min_chunk_bytes);

/*
 * Test hook: the next `count` kernel launches (of any entry point, after its
 * argument checks) return `status` -- NTS_ERR_CUDA, NTS_ERR_UNSUPPORTED or
 * NTS_ERR_TIMEOUT -- instead of launching, with nts_last_error() saying the
 * failure was injected; the device is not touched.  count = 0 turns the hook
 * off.  Lets callers' error handling be tested without a failing GPU.
 * Errors: INVALID_ARG for count < 0 or another status.
 */
NTS_API int nts_debug_inject_failure(int status, int count);

/*
 * The launch shape an MX request (T rows of D values, block size B, format
 * fmt, statistic p: 0 = RMSNorm, 1 or 2 = MXNorm) would get on a device
 * with `sm_count` SMs and `max_smem_optin` bytes of opt-in shared memory per
 * CTA, for a kernel of `regs` registers per thread (0: not limited by
 * registers; a launch uses the chosen kernel's own count), under the
 * current tuning, computed on the host without touching any device:
 * shape[0] units per thread (blocks, or halves of 64-value blocks),
 * shape[1] threads per row, shape[2] rows per tile, shape[3] ring stages,
 * shape[4] dynamic shared memory bytes.  Lets the launch rules be checked
 * exhaustively without a GPU.
 * Errors: INVALID_ARG for a bad query (regs outside 0..255 included);
 * UNSUPPORTED when no kernel serves it.
 */
NTS_API int nts_debug_mx_launch_shape(int64_t T, int64_t D, int B, int fmt, int p, int sm_count,
                                      int max_smem_optin, int regs, int32_t *shape);

/*
 * Programmatic dependent launch: 1 (default) = every kernel is launched with
 * programmatic stream serialization, so it may be scheduled while the grid
 * before it in the stream finishes (it waits for that grid's completion
 * before its first global-memory access); 0 = plain stream order.  Results
 * are identical either way.  Errors: INVALID_ARG for other values.
 */
NTS_API int nts_debug_set_pdl(int on);

/*
 * Test hook: every later launch tells its first ring stage to expect `bytes`
 * more than its copies deliver, so that stage's wait can only end by
 * expiring; the kernel then records NTS_ERR_TIMEOUT for nts_check_status and
 * returns with undefined outputs.  bytes must be a multiple of 16; 0 turns
 * the hook off.  Use with a short wait limit.
 */
NTS_API int nts_debug_set_missing_tx(uint32_t bytes);

/*
 * Self-check of the NVFP4 block scale (E4M3 code of fp32(amax/6), RNE,
 * saturating, and the fp32 reciprocal of its value) as the kernels form it:
 * the division by 6 by one multiply and two fmas (Brisebarre, Muller and
 * Raina, IEEE Trans. Computers 53(8), 2004) and the reciprocal from a
 * table.  Runs every non-negative fp32 absmax, 0 to +inf, on the current
 * device, blocking until done (a few ms), and returns
 *   *code_mismatches      absmaxes whose code or reciprocal differ from the
 *                         ones taken through the IEEE quotient and the IEEE
 *                         reciprocal (0 when the kernels are right);
 *   *quotient_mismatches  absmaxes with a normal quotient (>= 2^-126) where
 *                         the division differs from the IEEE quotient.
 * Errors: INVALID_ARG for NULL outputs, CUDA for a failed launch or copy.
 */
NTS_API int nts_debug_check_nvfp4_scale(uint64_t* code_mismatches, uint64_t* quotient_mismatches);

/*
 * Self-check of the E8M0 block exponent as the kernels form it (one add and
 * one shift: adding 0x4AFB0C to the fp32 bits of the normalized absmax
 * carries into the exponent field exactly when the significand rounds the
 * log2 up) against its definition field by field, for emax 8 (E4M3) and 2
 * (E2M1), over every non-negative fp32 absmax, 0 to +inf, on the current
 * device, blocking until done.  *mismatches = 0 when the kernels are right.
 * Errors: INVALID_ARG for a NULL output, CUDA for a failed launch or copy.
 */
NTS_API int nts_debug_check_e8m0(uint64_t* mismatches);

#ifdef __cplusplus
}
#endif

#endif /* NTS_DEBUG_H */
