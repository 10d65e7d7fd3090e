/*
 * moe_tail.h -- C ABI of the single-GPU decode-step MoE layer tail (libmoe_tail.so, sm_103a).
 *
 * The operation (one call, 1..max_rows token rows):
 *   1. residual add + RMSNorm:  s = x + residual;  r_new = bf16(s);
 *      n = bf16(r_new * rstd * gamma),  rstd = 1/sqrt(mean(r_new^2) + eps)
 *      -- "[AMD] integrate kimi k3 monokernel", Kernel Replacement table, row "The
 *         post-attention norm" (a fused add + RMSNorm kernel).
 *   2. router GEMV:  logits[r, e] = n[r, :] . W_r[e, :]  (bf16 inputs, fp32 accumulation)
 *      -- same table, row "The router".
 *   3. softmax + top-k + renormalisation (norm_topk_prob): the k experts with the largest
 *      logits, exact ties to the lowest expert id, in that pick order; weight of pick i =
 *      softmax restricted to the picked logits
 *      -- same table, row "The top-k"; section Refusals (norm_topk_prob is required);
 *         "glm53: Long-context indexer ..." page, Modifications table row 9 (top-8 tie
 *         shortcut: only an exact tie runs the id reduction, the pick order is unchanged).
 *   4. routed MXFP4 experts, each distinct expert streamed once per call:
 *      mid = bf16(SiLU(n . gate_j) * (n . up_j)),  y = mid . down
 *      -- Kernel Replacement row "The routed experts" (g1u1 = gate and up, SiLU);
 *         GLM-5.3 page, Modifications rows 16, 17, 20 (each expert once in up/gate and down).
 *   5. bf16 shared expert: ms = bf16(SiLU(n . Wg_j) * (n . Wu_j)),  ys = ms . Ws2
 *      -- Kernel Replacement rows "The shared expert gate_up / SiLU and mul / down".
 *   6. combine + residual update: out = bf16(sum over picks, in pick order, of
 *      w_i * y_i + ys);  residual <- r_new
 *      -- Kernel checks table (`out` and `res_out`).
 *
 * Storage formats (all row-major, contiguous, device memory, 16-byte aligned):
 *   bf16 values are IEEE bfloat16 bit patterns (uint16).
 *   MXFP4 (OCP): a row of K elements is K/2 code bytes (byte j: element 2j in the low
 *   nibble, 2j+1 in the high nibble; E2M1 codes) plus K/32 E8M0 scale bytes (2^(s-127)),
 *   scale b covering elements [32b, 32b+32).
 *
 * Return codes: 0 on success, a negative MOE_TAIL_ERR_* otherwise (moe_tail_strerror).
 * No entry point throws, aborts or prints.
 */
#ifndef MOE_TAIL_H
#define MOE_TAIL_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  MOE_TAIL_OK = 0,
  MOE_TAIL_ERR_INVALID_ARG = -1,   /* null/misaligned pointer, rows outside [1, max_rows] */
  MOE_TAIL_ERR_UNSUPPORTED = -2,   /* shape or option the library does not build */
  MOE_TAIL_ERR_CUDA = -3,          /* a CUDA call failed; moe_tail_last_cuda_error() */
  MOE_TAIL_ERR_TIMEOUT = -4,       /* a device-side wait ran past its budget */
  MOE_TAIL_ERR_NOT_CORESIDENT = -5,/* persistent mode cannot keep its whole grid resident */
  MOE_TAIL_ERR_DEVICE = -6         /* a device-side check failed (see moe_tail_get_status) */
};

/* Execution modes. */
enum {
  MOE_TAIL_MODE_MULTI_KERNEL = 0,  /* one launch per stage, stream-ordered */
  MOE_TAIL_MODE_PERSISTENT = 1     /* the whole call in one cooperative launch, one CTA per
                                      SM: add + RMSNorm, one grid-wide barrier (its
                                      generation word tags every call: nothing is reset
                                      between calls or graph replays), the router's parts
                                      spread over the CTAs, then the tensor-core expert roles
                                      of the multi-kernel form over the gate/up and then the
                                      down items, then the combine, handing over through the
                                      same per-expert and per-tile counts.  Bounded waits
                                      report MOE_TAIL_STATUS_TIMEOUT.  attn_dim must be 0
                                      (else MOE_TAIL_ERR_UNSUPPORTED at create) and the debug
                                      flags other than the stall injection do not apply.
                                      moe_tail_create returns MOE_TAIL_ERR_NOT_CORESIDENT when
                                      no CTA of it fits an SM; a launch that cannot keep every
                                      CTA resident fails with MOE_TAIL_ERR_CUDA instead of
                                      waiting. */
};

/* Bits of the device status word read by moe_tail_get_status (sticky until cleared). */
enum {
  /* A row's top-k found no number among its remaining logits (NaN router output): the
   * lowest untaken expert ids were picked for it. */
  MOE_TAIL_STATUS_BAD_ROUTING = 1,
  /* The distinct-expert count of a call fell outside [1, rows * top_k]. */
  MOE_TAIL_STATUS_BAD_DISTINCT = 2,
  /* A device-side wait ran past its budget; the kernel let its copies land and returned. */
  MOE_TAIL_STATUS_TIMEOUT = 4,
  /* A work item outside its matrix (or a misaligned shared-memory base) was skipped. */
  MOE_TAIL_STATUS_BAD_TILE = 8
};

/* debug_flags bits. */
enum {
  /* Run the expert stages with the warp-per-row CUDA-core kernels instead of the
   * TMA-streaming kernels (same results within the parity rule; for cross-checking). */
  MOE_TAIL_DEBUG_SIMPLE_KERNELS = 1,
  /* Launch every kernel as a plain stream-ordered launch (no programmatic dependent
   * launch overlap between consecutive kernels). */
  MOE_TAIL_DEBUG_NO_PDL = 2,
  /* Failure injection for tests: in the gate/up launch, the first CTA's producer leaves its
   * first pipeline stage unpublished, so that the consumers' bounded wait expires; the
   * kernel sets MOE_TAIL_STATUS_TIMEOUT in the status word and returns.  In the persistent
   * mode the first CTA never arrives at the grid barriers, so the others' waits expire the
   * same way.  The output of such a call is not meaningful. */
  MOE_TAIL_DEBUG_STALL_FIRST_STAGE = 4,
  /* Run the front (add + RMSNorm, router, top-k, dedup) as one launch in which every CTA
   * recomputes the row norms, instead of a norm launch followed by a router launch. */
  MOE_TAIL_DEBUG_FUSED_FRONT = 8,
  /* Run the expert stages on the TMA-streaming CUDA-core kernels (E2M1 weights converted to
   * f16 and fed to mma.sync with fp32 accumulation, E8M0 scales applied per 32-element
   * block) instead of the default tensor-core kernels.  The default form runs each routed
   * MXFP4 expert as tcgen05 block-scaled E2M1 x E2M1 MMAs whose activations enter as four
   * E2M1 planes with per-32 E8M0 scales (their sum approximates the bf16 activation to ~1e-3
   * of its block maximum), and the bf16 shared expert as tcgen05 bf16 MMAs, accumulating in
   * tensor memory ("glm53: Long-context indexer ..." page, Modifications row 16: every
   * using row a column of one multi-column product per expert).  Both forms meet the same
   * parity rule.  MOE_TAIL_DEBUG_FUSED_FRONT implies this form (the fused front writes no
   * activation planes). */
  MOE_TAIL_DEBUG_MMA_SYNC = 16,
  /* Tracing: every run records %globaltimer readings (nanoseconds) of its launches'
   * milestones into the handle (MOE_TAIL_TL_* slots below; zeroed by each run before its
   * first launch, which also keeps consecutive runs from overlapping), for
   * moe_tail_debug_timeline.  The stamps are recorded by the default expert form; slots of
   * stages a run does not have stay zero. */
  MOE_TAIL_DEBUG_TIMELINE = 32
};

/* Timeline slots: the first (or, for the ends, the last) reading of each milestone. */
enum {
  MOE_TAIL_TL_NORM_START = 0,        /* norm launch: first CTA past its wait on the previous */
  MOE_TAIL_TL_NORM_END = 1,          /* norm launch: last CTA done */
  MOE_TAIL_TL_ROUTER_START = 2,      /* router launch: first CTA past its wait */
  MOE_TAIL_TL_TOPK_START = 3,        /* router launch: its last CTA starts top-k and dedup */
  MOE_TAIL_TL_ROUTED = 4,            /* router launch: routing tables published */
  MOE_TAIL_TL_GATE_UP_START = 5,     /* gate/up launch: first CTA entered */
  MOE_TAIL_TL_GATE_UP_FIRST_COPY = 6,/* gate/up launch: first weight copy issued */
  MOE_TAIL_TL_GATE_UP_ROUTED = 7,    /* gate/up launch: first routed expert's copy issued */
  MOE_TAIL_TL_GATE_UP_END = 8,       /* gate/up launch: last CTA done */
  MOE_TAIL_TL_DOWN_START = 9,        /* down launch: first CTA entered */
  MOE_TAIL_TL_DOWN_FIRST_COPY = 10,  /* down launch: first weight copy issued */
  MOE_TAIL_TL_DOWN_END = 11,         /* down launch: last CTA done */
  MOE_TAIL_TL_COMBINE_START = 12,    /* combine launch: first CTA entered */
  MOE_TAIL_TL_COMBINE_END = 13,      /* combine launch: last output written */
  MOE_TAIL_TL_ROUTER_ALL_STARTED = 14, /* router launch: last CTA past its wait */
  MOE_TAIL_TL_GATE_UP_ALL_COPYING = 15,/* gate/up launch: last CTA's first weight copy issued */
  MOE_TAIL_TL_SLOTS = 16
};

typedef struct moe_tail moe_tail_t; /* opaque handle */

typedef struct {
  int32_t max_rows;       /* 1..32: the largest `rows` any run will pass; above 16 only the
                           * default expert form and the persistent mode, without attn_dim
                           * (the debug forms take 1..16; MOE_TAIL_ERR_UNSUPPORTED otherwise) */
  int32_t hidden;         /* H: multiple of 256 (of 512 above 2048), at most 32768 */
  int32_t n_experts;      /* E: 1..1024 */
  int32_t top_k;          /* k: 1..min(E, 32) */
  int32_t expert_inter;   /* I: multiple of 128 (of 512 above 2048) */
  int32_t shared_inter;   /* Is: multiple of 64 */
  float rms_eps;          /* RMSNorm epsilon (> 0) */
  int32_t norm_topk_prob; /* must be 1: the picked weights are renormalised to sum to 1 */
  int32_t mode;           /* MOE_TAIL_MODE_* */
  uint32_t wait_budget_us;/* budget of any device-side wait, microseconds; 0 = 100000 */
  uint32_t debug_flags;   /* 0 in production */
  int32_t attn_dim;       /* Ha: 0, or a multiple of 64 up to 65536 to put the attention
                           * output projection in front of the tail (moe_tail_run_attn) */
} moe_tail_config_t;

/* Weights are BORROWED device pointers: the caller keeps them alive and unmodified until
 * moe_tail_destroy.  The library never writes them.  One exception to reading them in place:
 * the default (tensor-core) expert form reads the routed experts' E8M0 scales (w13_scales,
 * w2_scales) from a copy made at create in the layout the block-scaled MMAs take them from
 * (groups of 4 blocks x 128 rows per 512 bytes), owned by the handle: 1/16 of the MXFP4 code
 * bytes, e.g. 352 MB for 256 experts at H 7168, I 2048.  A caller that changes those scales
 * after create calls moe_tail_refresh_scales before the next run. */
typedef struct {
  const void* gamma;       /* bf16 [H] */
  const void* router_w;    /* bf16 [E, H] */
  const void* w13_codes;   /* u8 [E, 2I, H/2]  rows [0, I) gate, [I, 2I) up */
  const void* w13_scales;  /* u8 E8M0 [E, 2I, H/32] */
  const void* w2_codes;    /* u8 [E, H, I/2] */
  const void* w2_scales;   /* u8 E8M0 [E, H, I/32] */
  const void* shared_w13;  /* bf16 [2Is, H]  rows [0, Is) gate, [Is, 2Is) up */
  const void* shared_w2;   /* bf16 [H, Is] */
  /* bf16 [H], or NULL.  When set, the shared expert's output enters the combine multiplied
   * by its row's gate sigmoid(n . shared_gate) ("[AMD] integrate kimi k3 monokernel" page,
   * Kernel Replacement row "shared expert gate, sigmoid and add").  Not available with
   * MOE_TAIL_DEBUG_FUSED_FRONT (refused at create). */
  const void* shared_gate;
  /* bf16 [H, Ha] when attn_dim > 0 (else NULL): the attention output projection of
   * moe_tail_run_attn ("[AMD] integrate kimi k3 monokernel" page, Kernel Replacement row 1,
   * a bf16 GEMM in front of the post-attention norm). */
  const void* out_proj;
} moe_tail_weights_t;

/* Validate the configuration and weights, allocate every scratch buffer the runs need on
 * the current CUDA device, and return a handle in *out.  Unsupported configurations are
 * refused here (MOE_TAIL_ERR_UNSUPPORTED), never at run time.  On error *out is NULL and
 * nothing is left allocated. */
int moe_tail_create(const moe_tail_config_t* cfg, const moe_tail_weights_t* w,
                    moe_tail_t** out);

/* Enqueue one call on `stream` (a cudaStream_t; NULL = legacy default stream).
 *   x        bf16 [rows, H] device, read only
 *   residual bf16 [rows, H] device, read and overwritten with bf16(x + residual)
 *   out      bf16 [rows, H] device, written with the MoE output
 * x, residual and out must not overlap.  The call allocates nothing, never synchronises
 * and is valid inside CUDA graph capture.  One stream at a time per handle: the handle's
 * scratch is reused by every call, so two calls on the same handle must be stream-ordered.
 * Device-side failures are reported by moe_tail_get_status, not by this return value. */
int moe_tail_run(moe_tail_t* h, const void* x, void* residual, void* out, int32_t rows,
                 void* stream);

/* The same call with the attention output projection in front (handles created with
 * attn_dim > 0; MOE_TAIL_ERR_UNSUPPORTED otherwise):
 *   attn     bf16 [rows, Ha] device, read-only, 16-byte aligned
 * x = bf16(attn . out_proj^T) (fp32 sums) is computed into the handle's scratch and the
 * tail runs on it exactly as moe_tail_run(x, residual, out) would. */
int moe_tail_run_attn(moe_tail_t* h, const void* attn, void* residual, void* out, int32_t rows,
                      void* stream);

/* The same call on HOST buffers; returns once out and residual hold the call's results.
 * Host memory the device reaches directly (16-byte aligned buffers: any host memory on a
 * device that uses the host's page tables, as on a Grace-Blackwell node over NVLink-C2C; else
 * page-locked memory, mapped into the device's address space) is read and written in place by
 * the call's kernels: x and residual read, out and residual written, no copy step (on a
 * non-default stream the first such call for a row count captures the call's launches as a
 * CUDA graph, so it must not run inside another capture, and every later one replays it with
 * its buffers passed through a page-locked argument block of the handle); the call's last
 * kernel then sets a page-locked completion word of the handle that this function polls
 * (the stream may still be retiring that kernel when it returns; if the call ends without
 * setting the word, a device-side failure reported by moe_tail_get_status, it returns once
 * the stream is idle).  Otherwise x and residual are copied to the handle's device staging
 * buffers, the call runs there, residual and out are copied back (one copy each way when the
 * buffers form one block [x; residual; out], residual_host = x_host + rows*H*2 bytes and
 * out_host = residual_host + rows*H*2), and `stream` is synchronised. */
int moe_tail_run_host(moe_tail_t* h, const void* x_host, void* residual_host, void* out_host,
                      int32_t rows, void* stream);

/* Synchronise the device and read the handle's device status word (0 = no failure).  A
 * nonzero word is sticky until moe_tail_clear_status (which, for a persistent-mode handle,
 * also resets the grid barrier a call that gave up may have left half counted). Returns
 * MOE_TAIL_ERR_DEVICE when the word is nonzero, MOE_TAIL_OK otherwise. */
int moe_tail_get_status(moe_tail_t* h, int32_t* device_status);

/* Guard check of the handle's scratch (for tests and debugging): every scratch buffer is
 * followed by 256 bytes of a fixed pattern written at create; this synchronises the device
 * and verifies them all.  Returns MOE_TAIL_OK, MOE_TAIL_ERR_DEVICE when a kernel wrote past
 * the end of a buffer (moe_tail_last_cuda_error() names the guard), MOE_TAIL_ERR_CUDA when
 * a copy fails, MOE_TAIL_ERR_INVALID_ARG for a NULL handle. */
int moe_tail_check_scratch(moe_tail_t* h);
int moe_tail_clear_status(moe_tail_t* h);

/* Copy the routing of the last run on `stream` (stream-ordered, synchronises it):
 * ids int32 [rows, k] and wts float [rows, k] in pick order, and the number of distinct
 * experts the call streamed.  Any output pointer may be NULL.  Host pointers. */
int moe_tail_debug_routing(moe_tail_t* h, int32_t* ids, float* wts, int32_t* n_distinct,
                           void* stream);

/* Optional per-stage timing.  When `events` is non-NULL, every later moe_tail_run records
 * events[2*i] before and events[2*i+1] after its stage i on the call's stream (stages in
 * launch order: add+RMSNorm, router, top-k+dedup, expert launches..., combine; see
 * moe_tail_launches_per_run).  The events are cudaEvent_t handles owned by the caller and
 * must outlive the runs that record them; n_events must be at least twice the launch
 * count.  NULL (or n_events = 0) turns the recording off.  The array is copied. */
int moe_tail_set_stage_events(moe_tail_t* h, void* const* events, int32_t n_events);

/* Number of kernels one moe_tail_run enqueues for `rows` rows (for launch accounting). */
int moe_tail_launches_per_run(const moe_tail_t* h, int32_t rows);

/* Routing of one call with no device allocation at all, for callers that cannot call
 * cudaMalloc: a host framework that owns every device allocation and hands a plugin only
 * its input and output tensors, or a decode step run from a memory pool that is frozen
 * once warm-up is over.  It runs add + RMSNorm, the router GEMV and the top-k with
 * renormalised weights on `stream`, with the arithmetic of the fused front
 * (MOE_TAIL_DEBUG_FUSED_FRONT): its logits are summed in another order than the default
 * front of moe_tail_run (which runs the router on the tensor cores), so they may differ in
 * the last bits, and a pick can differ from moe_tail_run's where two logits are that close.
 *   x, residual  bf16 [rows, hidden] device (both only read here)
 *   gamma bf16 [hidden], router_w bf16 [n_experts, hidden] device
 *   ids int32 [rows, top_k], wts float [rows, top_k] device, written in pick order;
 *   n_distinct int32 device, may be NULL: the number of distinct experts picked;
 *   status int32 device, may be NULL: this call's MOE_TAIL_STATUS_* bits (0 = clean;
 *     MOE_TAIL_STATUS_BAD_ROUTING when a row ran out of numeric logits, its remaining picks
 *     then being the lowest untaken ids), written when the call completes.
 * Its scratch is one fixed 71,696-byte array in the library's own device memory (a
 * file-scope variable that every GPU which loads the library keeps until the process
 * exits).  The array bounds the call: rows <= 16, n_experts <= 1024, top_k <= 32 (and
 * hidden a multiple of 128); anything larger returns MOE_TAIL_ERR_UNSUPPORTED.  The first
 * call on a device looks up the array's device address with that device current (once,
 * safe from several host threads).
 * Every call shares the array and it keeps the last call's contents (each call clears its
 * status word and counter first): calls that overlap on the same GPU race, so issue them
 * in one stream or otherwise ordered.  Nothing is allocated or freed.  The pages have no
 * counterpart to this entry point. */
int moe_tail_route_noalloc(const void* x, const void* residual, const void* gamma,
                           const void* router_w, int32_t rows, int32_t hidden,
                           int32_t n_experts, int32_t top_k, float rms_eps, int32_t* ids,
                           float* wts, int32_t* n_distinct, int32_t* status, void* stream);

/* The last run's timeline (handles created with MOE_TAIL_DEBUG_TIMELINE; otherwise
 * MOE_TAIL_ERR_UNSUPPORTED): synchronises the device and copies min(n, MOE_TAIL_TL_SLOTS)
 * stamps (uint64 nanoseconds of the GPU's global timer, 0 = milestone not reached) to the host
 * array `stamps`; returns the number copied, or a negative MOE_TAIL_ERR_*.  For tracing and
 * tests; the pages have no counterpart. */
int moe_tail_debug_timeline(moe_tail_t* h, uint64_t* stamps, int32_t n);

/* Re-make the handle's copy of w13_scales and w2_scales (see moe_tail_weights_t) from the
 * borrowed arrays, enqueued on `stream` (a cudaStream_t; NULL = legacy default stream):
 * later runs on that stream read the new scales.  A no-op returning MOE_TAIL_OK for forms
 * that read the scales in place (the debug forms, the persistent mode).  Returns
 * MOE_TAIL_ERR_INVALID_ARG for a NULL handle, MOE_TAIL_ERR_CUDA if the launch fails. */
int moe_tail_refresh_scales(moe_tail_t* h, void* stream);

/* Free the handle and its scratch (synchronises the device first).  NULL is a no-op. */
void moe_tail_destroy(moe_tail_t* h);

/* Static text for a return code. */
const char* moe_tail_strerror(int code);

/* Text of the last CUDA error seen by any entry point on this thread ("" if none). */
const char* moe_tail_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_TAIL_H */
