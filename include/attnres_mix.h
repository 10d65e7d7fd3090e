/*
 * attnres_mix.h -- C ABI of the AttnRes residual mix + RMSNorm for decode rows
 * (libmoe_tail.so, the second workload beside the MoE layer tail of moe_tail.h).
 *
 * Source: "Split the Kimi3 AttnRes mix across CTAs for decode rows" (voipmonitor/flare #11),
 * Description and commit message: one call of the mix adds the sublayer output into the
 * running sum of the current block (the prefix), commits a finished block, mixes the
 * row's sources with softmax weights from per-source dot and square-sum reductions, and
 * applies the RMSNorm to the mixture.  The page gives no formulas; the library computes,
 * for each row r (S = n_blocks + 1 sources):
 *
 *   prefix' = bf16(prefix + sub)                                  (residual add)
 *   v_0 .. v_{S-2} = blocks[0 .. n_blocks-1] of the row, v_{S-1} = prefix'
 *   score_i = (q . v_i) / sqrt(mean(v_i^2) + eps),  alpha = softmax(score)
 *   mix     = bf16(sum_i alpha_i v_i)
 *   y       = bf16(mix / sqrt(mean(mix^2) + eps) * gamma)           (RMSNorm of the mixture)
 *   commit != 0:  blocks[n_blocks] of the row = prefix', prefix = 0   (commit)
 *   commit == 0:  prefix = prefix'
 *
 * Arithmetic: fp32 sums and products; prefix' and the committed block are exact (the bf16
 * rounding of the exact sum); the CTAs of a row add their partials in one fixed order, so
 * a call's result does not depend on scheduling and a graph replay reproduces it bit for
 * bit.  Against an fp64 evaluation of the formulas the mixture may sit one bf16 step away
 * where the exact value is near a rounding boundary.  The CTAs of a row exchange their
 * partial sums through distributed shared memory; those waits are bounded and reported
 * through moe_attnres_mix_get_status.
 *
 * Return codes are those of moe_tail.h (MOE_TAIL_OK, MOE_TAIL_ERR_*; moe_tail_strerror and
 * moe_tail_last_cuda_error apply).
 */
#ifndef ATTNRES_MIX_H
#define ATTNRES_MIX_H

#include "moe_tail.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Launch flag: the launch may start while the previous kernel on the stream finishes
 * (programmatic dependent launch).  It then reads q and gamma at once, so the previous
 * kernel must not write them; everything else it reads, and everything it writes, waits
 * until the previous kernel has completed. */
#define MOE_ATTNRES_MIX_PDL 1u
/* Launch flag for failure tests only: one CTA of row 0 waits for a partial sum that never
 * comes.  Its wait gives up after the budget (50 ms), the device status word gets
 * MOE_TAIL_STATUS_TIMEOUT, and the call completes (its results are still right: the
 * awaited value is surplus). */
#define MOE_ATTNRES_MIX_DEBUG_STALL 2u

/* One call of the mix for `rows` rows of `hidden` columns, enqueued on `stream` (a
 * cudaStream_t; NULL is the legacy default stream).  Allocates nothing and never
 * synchronises; graph-capturable.
 *
 *   rows      1 .. 4096
 *   hidden    a multiple of 8 in [8, 65536]
 *   n_blocks  committed blocks, 0 .. 31 (S = n_blocks + 1 <= 32 sources)
 *   commit    nonzero: store prefix' as block n_blocks and zero the prefix
 *   eps       > 0, finite
 *   sub       device, bf16 [rows, hidden], read
 *   prefix    device, bf16 [rows, hidden], read and overwritten
 *   blocks    device, bf16 [n_blocks + (commit ? 1 : 0), rows, hidden]: block b of row r
 *             at element (b * rows + r) * hidden; blocks 0 .. n_blocks-1 read, block
 *             n_blocks written on a commit; may be NULL when n_blocks == 0 and commit == 0
 *   q         device, bf16 [hidden], the query of the scores
 *   gamma     device, bf16 [hidden], the RMSNorm weight
 *   mix, y    device, bf16 [rows, hidden], written
 *   flags     0 or MOE_ATTNRES_MIX_PDL (MOE_ATTNRES_MIX_DEBUG_STALL for failure tests)
 *
 * Every pointer is borrowed (the caller owns the memory) and must be 16-byte aligned.  The
 * outputs must not overlap q, gamma or blocks 0 .. n_blocks-1.
 * Errors (nothing is launched): MOE_TAIL_ERR_INVALID_ARG for rows, n_blocks or eps out of
 * range, a NULL or misaligned pointer, an unknown flag; MOE_TAIL_ERR_UNSUPPORTED for a
 * hidden size or source count outside the ranges above, or, for rows split into chunks
 * wider than 2048 columns (staged in shared memory), whose staging exceeds it
 * ((n_blocks + 5) * hidden / ctas_per_row * 2 bytes must stay under ~210 KB);
 * MOE_TAIL_ERR_CUDA when the launch fails. */
int moe_attnres_mix(int rows, int hidden, int n_blocks, int commit, float eps,
                    const void* sub, void* prefix, void* blocks, const void* q,
                    const void* gamma, void* mix, void* y, unsigned flags, void* stream);

/* The device status word of the mix on the current device (MOE_TAIL_STATUS_* bits; the
 * kernels OR MOE_TAIL_STATUS_TIMEOUT into it when an exchange between the CTAs of a row
 * waited past its 50 ms budget).  Synchronous: waits for the device's pending work.  Writes
 * the word to *status; clear != 0 zeroes it afterwards.  Returns MOE_TAIL_ERR_DEVICE when
 * the word was nonzero, MOE_TAIL_ERR_INVALID_ARG for a NULL status, MOE_TAIL_ERR_CUDA when
 * the copy fails, MOE_TAIL_OK otherwise. */
int moe_attnres_mix_get_status(int* status, int clear);

/* The CTAs (one thread-block cluster) that moe_attnres_mix gives each row for this shape:
 * 1, 2, 4 or 8; MOE_TAIL_ERR_UNSUPPORTED when the shape is not supported.  Host only. */
int moe_attnres_mix_ctas_per_row(int hidden, int n_blocks);

#ifdef __cplusplus
}
#endif

#endif /* ATTNRES_MIX_H */
