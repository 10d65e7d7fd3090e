// moe_tail_api.cu -- the C ABI of libmoe_tail.so: configuration checks, scratch
// ownership, and the stream-ordered sequence of kernel launches of one call.
//
// The refusal of unsupported configurations at creation follows the Refusals section of
// the "[AMD] integrate kimi k3 monokernel" page (the layer stops at startup, never at run
// time); the borrowed weights follow its remark that the kernels read the weights in
// place and copy none; scratch is owned per handle and reused by every call.
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <chrono>
#include <new>

#include <math.h>

#include "attnres_mix.h"
#include "k_mix.cuh"
#include "k_persist.cuh"
#include "moe_tail.h"
#include "moe_tail_internal.cuh"

using namespace mtail;

// Every scratch buffer is followed by kCanaryBytes of a known pattern; a kernel that writes
// past the end of a buffer changes them (moe_tail_check_scratch).
constexpr int kMaxCanaries = 32;
constexpr size_t kCanaryBytes = 256;
constexpr unsigned char kCanaryByte = 0xA5;

struct moe_tail {
  moe_tail_config_t cfg;
  Weights w;
  StreamMaps maps;     // TMA descriptors of the streamed weights
  TcMaps tcmaps;       // and of the tensor-core form (the default expert stages)
  Scratch s;
  void* slab;          // one device allocation holding every scratch buffer
  size_t slab_bytes;
  void* stage;         // device staging for moe_tail_run_host: x, residual, out
  void* atoms;         // the tensor-core form's copy of w13s and w2s in scale-factor atoms
  int host_direct;     // the device reads pageable host memory through the host's page tables
  uint32_t* hdone;     // page-locked completion word of moe_tail_run_host (mapped), or null
  uint32_t* hdone_dev; // its device address
  uint32_t hseq;       // the last value a call asked for in it
  HostArgs* hargs;     // page-locked arguments of the host-buffer call (mapped, after hdone)
  HostArgs* hargs_dev; // their device address
  // moe_tail_run_host on a non-default stream: one graph per row count of the call's launches,
  // which take the buffers from hargs
  cudaGraph_t hgraph[kMaxRows + 1];
  cudaGraphExec_t hexec[kMaxRows + 1];
  int device;
  int num_sms;
  int persist_grid;    // CTAs of the single persistent launch (MOE_TAIL_MODE_PERSISTENT)
  int last_rows;
  cudaEvent_t ev[2 * 16];  // optional stage events (moe_tail_set_stage_events)
  int n_ev;
  size_t canary_off[kMaxCanaries];  // slab offsets of the guard words after each buffer
  int n_canary;
};

static thread_local char g_cuda_err[256];

static int cuda_fail(cudaError_t e) {
  snprintf(g_cuda_err, sizeof(g_cuda_err), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
  return MOE_TAIL_ERR_CUDA;
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

extern "C" const char* moe_tail_strerror(int code) {
  switch (code) {
    case MOE_TAIL_OK: return "ok";
    case MOE_TAIL_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, rows out of range)";
    case MOE_TAIL_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_TAIL_ERR_CUDA: return "CUDA error";
    case MOE_TAIL_ERR_TIMEOUT: return "device-side wait exceeded its budget";
    case MOE_TAIL_ERR_NOT_CORESIDENT: return "persistent grid cannot be co-resident";
    case MOE_TAIL_ERR_DEVICE: return "device-side check failed";
    default: return "unknown error";
  }
}

extern "C" const char* moe_tail_last_cuda_error(void) { return g_cuda_err; }

static_assert(MOE_TAIL_DEBUG_STALL_FIRST_STAGE == (int)kDebugStallFirstStage,
              "debug bit values agree");
static_assert(MOE_TAIL_DEBUG_MMA_SYNC == (int)kDebugMmaSync, "debug bit values agree");
static_assert(MOE_TAIL_DEBUG_TIMELINE == (int)kDebugTimeline, "debug bit values agree");
static_assert(MOE_TAIL_TL_SLOTS == (int)kTlSlots, "timeline slots agree");

// The expert stages run on the tcgen05 kernels unless a debug flag picks another form (the
// mma.sync streaming kernels, the cross-checking CUDA-core kernels, or the fused front, which
// writes no activation planes); the persistent launch runs them too (its debug flags other
// than the stall injection do not apply).
static bool uses_tc(const moe_tail_config_t* c) {
  if (c->mode == MOE_TAIL_MODE_PERSISTENT) return true;
  return c->mode == MOE_TAIL_MODE_MULTI_KERNEL &&
         !(c->debug_flags & (MOE_TAIL_DEBUG_MMA_SYNC | MOE_TAIL_DEBUG_SIMPLE_KERNELS |
                             MOE_TAIL_DEBUG_FUSED_FRONT));
}

static int check_config(const moe_tail_config_t* c) {
  if (c->max_rows < 1 || c->max_rows > kMaxRows) return MOE_TAIL_ERR_UNSUPPORTED;
  // more than 16 rows: the default expert form only, without the out_proj stage (whose
  // streaming launch keeps 16-row register tiles)
  if (c->max_rows > kMaxRowsOther && (!uses_tc(c) || c->attn_dim != 0))
    return MOE_TAIL_ERR_UNSUPPORTED;
  // hidden: whole 256-element stages; above 2048 the E8M0 rows (hidden/32 bytes) must be
  // whole 16-byte units for the scale-window tensor maps of the CUDA-core form
  if (c->hidden < 256 || c->hidden % 256) return MOE_TAIL_ERR_UNSUPPORTED;
  if (c->hidden > 2048 && c->hidden % 512) return MOE_TAIL_ERR_UNSUPPORTED;
  if (c->hidden > (1 << 15)) return MOE_TAIL_ERR_UNSUPPORTED;
  if (c->n_experts < 1 || c->n_experts > kMaxExperts) return MOE_TAIL_ERR_UNSUPPORTED;
  if (c->top_k < 1 || c->top_k > kMaxTopK || c->top_k > c->n_experts)
    return MOE_TAIL_ERR_UNSUPPORTED;
  if (c->expert_inter < 128 || c->expert_inter % 128 || c->expert_inter > (1 << 16))
    return MOE_TAIL_ERR_UNSUPPORTED;
  if (c->expert_inter > 2048 && c->expert_inter % 512) return MOE_TAIL_ERR_UNSUPPORTED;
  if (c->shared_inter < 64 || c->shared_inter % 64 || c->shared_inter > (1 << 16))
    return MOE_TAIL_ERR_UNSUPPORTED;
  if (!(c->rms_eps > 0.f)) return MOE_TAIL_ERR_UNSUPPORTED;
  if (c->attn_dim < 0 || c->attn_dim > (1 << 16) || c->attn_dim % 64)
    return MOE_TAIL_ERR_UNSUPPORTED;
  if (c->norm_topk_prob != 1) return MOE_TAIL_ERR_UNSUPPORTED;
  if (c->mode != MOE_TAIL_MODE_MULTI_KERNEL && c->mode != MOE_TAIL_MODE_PERSISTENT)
    return MOE_TAIL_ERR_UNSUPPORTED;
  // the persistent launch covers the tail from x on (no out_proj stage in front of it)
  if (c->mode == MOE_TAIL_MODE_PERSISTENT && c->attn_dim != 0) return MOE_TAIL_ERR_UNSUPPORTED;

  return MOE_TAIL_OK;
}

// Carve the scratch buffers out of one slab (256-byte aligned pieces, each followed by a
// guard region whose offset goes to canaries[]).
static size_t carve(const moe_tail_config_t* c, char* base, Scratch* s, size_t* canaries,
                    int* n_canary) {
  const size_t R = c->max_rows, H = c->hidden, E = c->n_experts, k = c->top_k,
               I = c->expert_inter, Is = c->shared_inter, P = R * k;
  size_t off = 0;
  int nc = 0;
  auto take = [&](size_t bytes) -> char* {
    char* p = base ? base + off : nullptr;
    off += (bytes + 255) & ~(size_t)255;
    if (nc < kMaxCanaries) {
      if (canaries) canaries[nc] = off;
      ++nc;
    }
    off += kCanaryBytes;
    return p;
  };
  s->rnew = (__nv_bfloat16*)take(R * H * 2);
  s->n = (__nv_bfloat16*)take(R * H * 2);
  s->n16 = (__half*)take(R * H * 2);
  s->n16s = (float*)take(R * 4);
  s->logits = (float*)take(R * E * 4);
  s->logit_parts = (float*)take((size_t)router_max_parts() * R * E * 4);
  s->ids = (int32_t*)take(P * 4);
  s->wts = (float*)take(P * 4);
  s->n_distinct = (int32_t*)take(4);
  s->uniq = (int32_t*)take(P * 4);
  s->user_off = (int32_t*)take((P + 1) * 4);
  s->user_list = (int32_t*)take(P * 4);
  s->mid = (__nv_bfloat16*)take(P * I * 2);
  s->mid16 = (__half*)take(P * I * 2);
  s->mid16s = (float*)take(P * (I / 32) * 4);
  s->ms = (__nv_bfloat16*)take(R * Is * 2);
  s->y = (float*)take(P * H * 4);
  s->ys = (float*)take(R * H * 4);
  s->sgate = (float*)take(R * 4);
  s->gate_part = (float*)take(R * kMaxNormParts * 4);
  s->xproj = (__nv_bfloat16*)take(R * H * 2);
  s->xpart = (float*)take((size_t)kMaxOutProjParts * R * H * 4);
  s->gpart = (float*)take((size_t)std::min<size_t>(Is / 64, kMaxSharedSplitItems) *
                          kMaxSharedParts * 128 * R * 4);
  s->np4 = (uint8_t*)take(4 * R * H / 2);
  s->np4a = (uint8_t*)take((size_t)sf_atoms_per_tile((int)H) * 512);
  s->mid4 = (uint8_t*)take(4 * P * I / 2);
  s->mid4a = (uint8_t*)take(std::min<size_t>(E, P) * sf_atoms_per_tile((int)I) * 512);
  s->tl = (c->debug_flags & MOE_TAIL_DEBUG_TIMELINE) ? (unsigned long long*)take(kTlSlots * 8)
                                                     : nullptr;
  s->status = (int32_t*)take(4);
  s->counters = (uint32_t*)take(kCtrWords * 4);
  if (n_canary) *n_canary = nc < kMaxCanaries ? nc : kMaxCanaries;
  return off;
}

extern "C" int moe_tail_create(const moe_tail_config_t* cfg, const moe_tail_weights_t* w,
                               moe_tail_t** out) {
  if (!out) return MOE_TAIL_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg || !w) return MOE_TAIL_ERR_INVALID_ARG;
  int rc = check_config(cfg);
  if (rc) return rc;
  const void* ptrs[8] = {w->gamma, w->router_w, w->w13_codes, w->w13_scales,
                         w->w2_codes, w->w2_scales, w->shared_w13, w->shared_w2};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return MOE_TAIL_ERR_INVALID_ARG;
  if (w->shared_gate && !aligned16(w->shared_gate)) return MOE_TAIL_ERR_INVALID_ARG;
  // out_proj exactly when the configuration asks for it
  if ((cfg->attn_dim > 0) != (w->out_proj != nullptr)) return MOE_TAIL_ERR_INVALID_ARG;
  if (w->out_proj && !aligned16(w->out_proj)) return MOE_TAIL_ERR_INVALID_ARG;
  // the fused front computes n chunk by chunk across CTAs: it has no row-wide gate reduction
  if (w->shared_gate && (cfg->debug_flags & MOE_TAIL_DEBUG_FUSED_FRONT))
    return MOE_TAIL_ERR_UNSUPPORTED;

  moe_tail_t* h = new (std::nothrow) moe_tail_t;
  if (!h) return MOE_TAIL_ERR_CUDA;
  memset(h, 0, sizeof(*h));
  h->cfg = *cfg;
  h->w.gamma = (const __nv_bfloat16*)w->gamma;
  h->w.w_r = (const __nv_bfloat16*)w->router_w;
  h->w.w13c = (const uint8_t*)w->w13_codes;
  h->w.w13s = (const uint8_t*)w->w13_scales;
  h->w.w2c = (const uint8_t*)w->w2_codes;
  h->w.w2s = (const uint8_t*)w->w2_scales;
  h->w.ws13 = (const __nv_bfloat16*)w->shared_w13;
  h->w.ws2 = (const __nv_bfloat16*)w->shared_w2;
  h->w.wsg = (const __nv_bfloat16*)w->shared_gate;
  h->w.wo = (const __nv_bfloat16*)w->out_proj;

  cudaError_t e = cudaGetDevice(&h->device);
  if (e == cudaSuccess) e = prepare_stream_kernels();
  if (e == cudaSuccess) e = prepare_front_kernels();
  if (e == cudaSuccess && uses_tc(cfg)) e = prepare_stream_tc_kernels();
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&h->host_direct, cudaDevAttrPageableMemoryAccessUsesHostPageTables,
                               h->device);
  if (e == cudaSuccess && cfg->mode == MOE_TAIL_MODE_PERSISTENT)
    h->persist_grid = h->num_sms;  // one CTA per SM (checked once the layout is known)
  if (e != cudaSuccess) { delete h; return cuda_fail(e); }
  h->slab_bytes = carve(cfg, nullptr, &h->s, nullptr, nullptr);
  e = cudaMalloc(&h->slab, h->slab_bytes);
  if (e != cudaSuccess) { delete h; return cuda_fail(e); }
  carve(cfg, (char*)h->slab, &h->s, h->canary_off, &h->n_canary);
  const size_t act = (size_t)cfg->max_rows * cfg->hidden * 2;
  e = cudaMalloc(&h->stage, 3 * act);
  if (e == cudaSuccess) e = cudaMemset(h->slab, 0, h->slab_bytes);
  for (int i = 0; e == cudaSuccess && i < h->n_canary; ++i)
    e = cudaMemset((char*)h->slab + h->canary_off[i], kCanaryByte, kCanaryBytes);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    cudaFree(h->slab);
    if (h->stage) cudaFree(h->stage);
    delete h;
    return cuda_fail(e);
  }
  {
    Dims d0;
    d0.R = cfg->max_rows; d0.Rmax = cfg->max_rows; d0.H = cfg->hidden; d0.E = cfg->n_experts;
    d0.k = cfg->top_k; d0.I = cfg->expert_inter; d0.Is = cfg->shared_inter; d0.eps = cfg->rms_eps;
    d0.Ha = cfg->attn_dim;
    d0.Pk = 1;
    if (uses_tc(cfg)) {
      // the routed experts' E8M0 scales in the atoms the tensor-core kernels copy per stage
      e = cudaMalloc(&h->atoms, scale_atom_bytes(d0));
      if (e == cudaSuccess) {
        h->w.w13a = (const uint8_t*)h->atoms;
        h->w.w2a = (const uint8_t*)h->atoms +
                   (size_t)d0.E * (d0.I / 64) * sf_atoms_per_tile(d0.H) * 512;
        e = launch_scale_atoms(d0, h->w, (uint8_t*)h->atoms, 0);
      }
      if (e == cudaSuccess) e = cudaDeviceSynchronize();
      if (e != cudaSuccess) {
        cudaFree(h->slab);
        cudaFree(h->stage);
        if (h->atoms) cudaFree(h->atoms);
        delete h;
        return cuda_fail(e);
      }
    }
    int mrc = make_stream_maps(&h->maps, d0, h->w, h->s);
    int limit = kSmemLimit;
    if (mrc == 0 && cfg->mode == MOE_TAIL_MODE_PERSISTENT) {
      const TcLayout l0 = make_tc_layout(d0.Rmax, d0.k, kSmemLimit);
      if (persistent_smem_limit(l0.nmax, &limit) != cudaSuccess) mrc = -3;
    }
    if (mrc == 0 && uses_tc(cfg))
      mrc = make_tc_maps(&h->tcmaps, h->maps, d0, h->w, h->s, limit);
    if (mrc == 0 && cfg->mode == MOE_TAIL_MODE_PERSISTENT) {
      // every CTA of the cooperative launch resident at once: one per SM
      int per_sm = 0;
      if (persistent_prepare(h->tcmaps, &per_sm) != cudaSuccess) mrc = -3;
      else if (per_sm < 1) mrc = -4;
    }
    if (mrc != 0) {
      cudaFree(h->slab);
      cudaFree(h->stage);
      if (h->atoms) cudaFree(h->atoms);
      delete h;
      if (mrc == -1) {
        snprintf(g_cuda_err, sizeof(g_cuda_err), "no cuTensorMapEncodeTiled");
        return MOE_TAIL_ERR_CUDA;
      }
      if (mrc == -3) return cuda_fail(cudaGetLastError());
      if (mrc == -4) return MOE_TAIL_ERR_NOT_CORESIDENT;
      return MOE_TAIL_ERR_UNSUPPORTED;
    }
  }
  *out = h;
  return MOE_TAIL_OK;
}

extern "C" int moe_tail_set_stage_events(moe_tail_t* h, void* const* events, int32_t n_events) {
  if (!h || n_events < 0) return MOE_TAIL_ERR_INVALID_ARG;
  if (!events || n_events == 0) { h->n_ev = 0; return MOE_TAIL_OK; }
  if (n_events > 2 * 16) n_events = 2 * 16;
  for (int i = 0; i < n_events; ++i) {
    if (!events[i]) return MOE_TAIL_ERR_INVALID_ARG;
    h->ev[i] = (cudaEvent_t)events[i];
  }
  h->n_ev = n_events;
  return MOE_TAIL_OK;
}

extern "C" int moe_tail_launches_per_run(const moe_tail_t* h, int32_t rows) {
  (void)rows;
  if (!h) return 0;
  if (h->cfg.mode == MOE_TAIL_MODE_PERSISTENT) return 1;
  if (h->cfg.debug_flags & MOE_TAIL_DEBUG_SIMPLE_KERNELS) return 8;
  return (h->cfg.debug_flags & MOE_TAIL_DEBUG_FUSED_FRONT) ? 4 : 5;
}

// One call: x is the tail's input, or null with attn the attention output to project first;
// done, seq: a host-visible word the call's last kernel sets to seq when its outputs are
// visible to the host (null: none); ha: the tensor-core forms take x, residual, out and seq
// from a host-buffer call's arguments at run time instead (null: as given).
static int run_impl(moe_tail_t* h, const void* x, const void* attn, void* residual, void* out,
                    int32_t rows, void* stream, uint32_t* done = nullptr, uint32_t seq = 0u,
                    const HostArgs* ha = nullptr) {
  cudaStream_t st = (cudaStream_t)stream;
  Dims d;
  d.R = rows;
  d.Rmax = h->cfg.max_rows;
  d.H = h->cfg.hidden;
  d.E = h->cfg.n_experts;
  d.k = h->cfg.top_k;
  d.I = h->cfg.expert_inter;
  d.Is = h->cfg.shared_inter;
  d.Ha = h->cfg.attn_dim;
  d.Pk = 1;
  d.eps = h->cfg.rms_eps;
  cudaError_t e;
  int stage_i = 0;
  auto mark = [&](int which) -> cudaError_t {
    const int idx = 2 * stage_i + which;
    if (idx < h->n_ev) return cudaEventRecord(h->ev[idx], st);
    return cudaSuccess;
  };
#define MT_STAGE(call)                                  \
  do {                                                  \
    if ((e = mark(0))) return cuda_fail(e);             \
    if ((e = (call))) return cuda_fail(e);              \
    if ((e = mark(1))) return cuda_fail(e);             \
    ++stage_i;                                          \
  } while (0)
  const bool pdl = !(h->cfg.debug_flags & MOE_TAIL_DEBUG_NO_PDL);
  const bool simple = (h->cfg.debug_flags & MOE_TAIL_DEBUG_SIMPLE_KERNELS) != 0;
  const bool tc = uses_tc(&h->cfg);
  const uint64_t budget_ns =
      (uint64_t)(h->cfg.wait_budget_us ? h->cfg.wait_budget_us : 100000u) * 1000ull;
  const float* xpart = nullptr;
  if (h->s.tl && (e = cudaMemsetAsync(h->s.tl, 0, kTlSlots * 8, st))) return cuda_fail(e);
  if (h->cfg.mode == MOE_TAIL_MODE_PERSISTENT) {
    // the whole call in one cooperative launch (such a handle has no out_proj stage)
    MT_STAGE(launch_persistent(h->tcmaps, d, (const __nv_bfloat16*)x, (__nv_bfloat16*)residual,
                               (__nv_bfloat16*)out, h->w, h->s, h->persist_grid, budget_ns,
                               (h->cfg.debug_flags & MOE_TAIL_DEBUG_STALL_FIRST_STAGE) != 0, st,
                               done, seq, ha));
    h->last_rows = rows;
    return MOE_TAIL_OK;
  }
  if (attn) {
    // the attention output projection into scratch; the call's map of attn travels with
    // the launch's parameters (a graph replays it as captured).  Each 128-output box is
    // split along K into 1, 2, 4 or 8 parts, whose fp32 sums the norm launch adds in part
    // order; the count taken is the one whose busiest CTA streams the fewest K columns
    // (ceil(items / SMs) items of Ha / parts columns; ties keep the smaller count).  The
    // fused front reads x whole, so it takes one part.
    StreamMaps m = h->maps;
    const int mrc = make_attn_map(&m, attn, rows, d);
    if (mrc) return mrc == -1 ? cuda_fail(cudaErrorNotSupported) : MOE_TAIL_ERR_INVALID_ARG;
    int pk = 1;
    if (!(h->cfg.debug_flags & MOE_TAIL_DEBUG_FUSED_FRONT)) {
      const long boxes = d.H / 128;
      long best = -1;
      for (int p = 1; p <= kMaxOutProjParts; p <<= 1) {
        if ((d.Ha / 64) % p) continue;
        const long cols = (boxes * p + h->num_sms - 1) / h->num_sms * (d.Ha / p);
        if (best < 0 || cols < best) { best = cols; pk = p; }
      }
    }
    d.Pk = pk;
    MT_STAGE(launch_stream(2, m, d, h->w, h->s, h->num_sms, budget_ns, st, pdl,
                           h->cfg.debug_flags));
    x = h->s.xproj;
    if (pk > 1) xpart = h->s.xpart;
  }
  if (simple) {
    MT_STAGE(launch_add_rmsnorm(d, (const __nv_bfloat16*)x, (const __nv_bfloat16*)residual,
                                h->w, h->s, st, pdl, xpart));
    MT_STAGE(launch_router(d, h->w, h->s, st, pdl));
    MT_STAGE(launch_topk_dedup(d, h->s, st, pdl));
    MT_STAGE(launch_experts_simple(d, h->w, h->s, h->num_sms, st));
  } else {
    if (h->cfg.debug_flags & MOE_TAIL_DEBUG_FUSED_FRONT) {
      MT_STAGE(launch_front_fused(d, (const __nv_bfloat16*)x, (const __nv_bfloat16*)residual,
                                  h->w, h->s, st, pdl));
    } else {
      MT_STAGE(launch_add_rmsnorm(d, (const __nv_bfloat16*)x, (const __nv_bfloat16*)residual,
                                  h->w, h->s, st, pdl, xpart, tc, ha));
      MT_STAGE(launch_router_topk(d, h->w, h->s, st, pdl));
    }
    const uint32_t dbg = h->cfg.debug_flags;
    if (tc) {
      MT_STAGE(launch_stream_tc(0, h->tcmaps, d, h->w, h->s, h->num_sms, budget_ns, st, pdl, dbg));
      MT_STAGE(launch_stream_tc(1, h->tcmaps, d, h->w, h->s, h->num_sms, budget_ns, st, pdl, dbg));
    } else {
      MT_STAGE(launch_stream(0, h->maps, d, h->w, h->s, h->num_sms, budget_ns, st, pdl, dbg));
      MT_STAGE(launch_stream(1, h->maps, d, h->w, h->s, h->num_sms, budget_ns, st, pdl, dbg));
    }
  }
  // after the streaming kernels the combine waits per 128 outputs for the down items that
  // write them; after the cross-checking kernels it waits for the previous launch
  MT_STAGE(launch_combine(d, h->s, (__nv_bfloat16*)out, (__nv_bfloat16*)residual, st, pdl,
                          !simple, budget_ns, h->w.wsg != nullptr, done, seq, ha,
                          tc ? h->num_sms : 0));
#undef MT_STAGE
  h->last_rows = rows;
  return MOE_TAIL_OK;
}

extern "C" int moe_tail_run(moe_tail_t* h, const void* x, void* residual, void* out,
                            int32_t rows, void* stream) {
  if (!h || !x || !residual || !out) return MOE_TAIL_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(residual) || !aligned16(out)) return MOE_TAIL_ERR_INVALID_ARG;
  if (rows < 1 || rows > h->cfg.max_rows) return MOE_TAIL_ERR_INVALID_ARG;
  return run_impl(h, x, nullptr, residual, out, rows, stream);
}

extern "C" int moe_tail_run_attn(moe_tail_t* h, const void* attn, void* residual, void* out,
                                 int32_t rows, void* stream) {
  if (!h || !attn || !residual || !out) return MOE_TAIL_ERR_INVALID_ARG;
  if (!aligned16(attn) || !aligned16(residual) || !aligned16(out))
    return MOE_TAIL_ERR_INVALID_ARG;
  if (rows < 1 || rows > h->cfg.max_rows) return MOE_TAIL_ERR_INVALID_ARG;
  if (h->cfg.attn_dim <= 0) return MOE_TAIL_ERR_UNSUPPORTED;
  return run_impl(h, nullptr, attn, residual, out, rows, stream);
}

// The device address of a page-locked host buffer, or null (pageable memory).  Page-locked
// memory is mapped into the device's address space (unified addressing), so kernels read and
// write it in place: over NVLink-C2C on a Grace-Blackwell node.
static void* mapped_host(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // pageable memory may report an error on some drivers: not sticky
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost) return nullptr;
  return a.devicePointer;
}

extern "C" int moe_tail_run_host(moe_tail_t* h, const void* x_host, void* residual_host,
                                 void* out_host, int32_t rows, void* stream) {
  if (!h || !x_host || !residual_host || !out_host) return MOE_TAIL_ERR_INVALID_ARG;
  if (rows < 1 || rows > h->cfg.max_rows) return MOE_TAIL_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  const size_t bytes = (size_t)rows * h->cfg.hidden * 2;
  // device staging [x; residual; out], `bytes` apart, so that host buffers laid out the
  // same way move in one copy each way
  char* dx = (char*)h->stage;
  char* dres = dx + bytes;
  char* dout = dres + bytes;
  const bool in_block = (const char*)residual_host == (const char*)x_host + bytes;
  const bool out_block = (char*)out_host == (char*)residual_host + bytes;
  cudaError_t e;
  {
    // host memory the device reaches directly (any host memory where the device uses the
    // host's page tables, else page-locked buffers): the call's kernels read x and the
    // residual and write out and the residual in place, no copy step
    void* mx = h->host_direct ? (void*)x_host : mapped_host(x_host);
    void* mr = h->host_direct ? residual_host : mx ? mapped_host(residual_host) : nullptr;
    void* mo = h->host_direct ? out_host : mr ? mapped_host(out_host) : nullptr;
    if (mo && aligned16(mx) && aligned16(mr) && aligned16(mo)) {
      // the call's last kernel writes its number to a page-locked word once the outputs are
      // visible to the host; the host polls that word (and, every 20 us or so, the stream,
      // which ends the wait if the call finished without writing it: a device-side failure,
      // reported by moe_tail_get_status).  The stream is queried rarely: a query costs the
      // polling thread about a microsecond, during which the word's arrival goes unseen.
      if (!h->hdone) {
        void* pg = nullptr;
        e = cudaHostAlloc(&pg, 128, cudaHostAllocMapped);
        void* dg = nullptr;
        if (e == cudaSuccess) e = cudaHostGetDevicePointer(&dg, pg, 0);
        if (e != cudaSuccess) {
          if (pg) cudaFreeHost(pg);
          return cuda_fail(e);
        }
        h->hdone = (uint32_t*)pg;
        h->hdone_dev = (uint32_t*)dg;
        h->hargs = (HostArgs*)((char*)pg + 64);
        h->hargs_dev = (HostArgs*)((char*)dg + 64);
        __atomic_store_n(h->hdone, 0u, __ATOMIC_RELEASE);
      }
      const uint32_t seq = ++h->hseq ? h->hseq : ++h->hseq;  // never 0 (the initial value)
      // the tensor-core forms on a non-default stream: a graph of the call's launches,
      // captured once per row count, reads this call's buffers and number from hargs
      const bool graph = uses_tc(&h->cfg) && h->n_ev == 0 && h->cfg.attn_dim == 0 &&
                         st != nullptr && st != cudaStreamLegacy && st != cudaStreamPerThread;
      if (graph) {
        if (!h->hexec[rows]) {
          e = cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal);
          if (e != cudaSuccess) return cuda_fail(e);
          const int rc = run_impl(h, nullptr, nullptr, nullptr, nullptr, rows, stream,
                                  h->hdone_dev, 0u, h->hargs_dev);
          cudaGraph_t g = nullptr;
          e = cudaStreamEndCapture(st, &g);
          if (e == cudaSuccess && rc != MOE_TAIL_OK) e = cudaErrorUnknown;
          cudaGraphExec_t ex = nullptr;
          if (e == cudaSuccess) e = cudaGraphInstantiate(&ex, g, 0);
          if (e != cudaSuccess) {
            if (g) cudaGraphDestroy(g);
            return rc != MOE_TAIL_OK ? rc : cuda_fail(e);
          }
          h->hgraph[rows] = g;
          h->hexec[rows] = ex;
        }
      }
      // the kernels take the buffers and the call number from the argument block (written
      // before the launch; the previous call has finished reading it)
      h->hargs->x = mx;
      h->hargs->residual = mr;
      h->hargs->out = mo;
      h->hargs->seq = seq;
      __atomic_thread_fence(__ATOMIC_SEQ_CST);
      if (graph) {
        e = cudaGraphLaunch(h->hexec[rows], st);
        if (e != cudaSuccess) return cuda_fail(e);
        h->last_rows = rows;
      } else {
        const int rc = run_impl(h, mx, nullptr, mr, mo, rows, stream, h->hdone_dev, seq,
                                uses_tc(&h->cfg) && h->cfg.attn_dim == 0 ? h->hargs_dev : nullptr);
        if (rc) return rc;
      }
      auto last = std::chrono::steady_clock::now();
      for (uint32_t i = 1; __atomic_load_n(h->hdone, __ATOMIC_ACQUIRE) != seq; ++i) {
        if ((i & 63) == 0) {
          const auto now = std::chrono::steady_clock::now();
          if (now - last < std::chrono::microseconds(20)) continue;
          last = now;
          e = cudaStreamQuery(st);
          if (e == cudaSuccess) break;
          if (e != cudaErrorNotReady) return cuda_fail(e);
        }
      }
      return MOE_TAIL_OK;
    }
  }
  if (in_block) {
    e = cudaMemcpyAsync(dx, x_host, 2 * bytes, cudaMemcpyHostToDevice, st);
  } else {
    e = cudaMemcpyAsync(dx, x_host, bytes, cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dres, residual_host, bytes, cudaMemcpyHostToDevice, st);
  }
  if (e != cudaSuccess) return cuda_fail(e);
  int rc = moe_tail_run(h, dx, dres, dout, rows, stream);
  if (rc) return rc;
  if (out_block) {
    e = cudaMemcpyAsync(residual_host, dres, 2 * bytes, cudaMemcpyDeviceToHost, st);
  } else {
    e = cudaMemcpyAsync(residual_host, dres, bytes, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(out_host, dout, bytes, cudaMemcpyDeviceToHost, st);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return e == cudaSuccess ? MOE_TAIL_OK : cuda_fail(e);
}

extern "C" int moe_tail_get_status(moe_tail_t* h, int32_t* device_status) {
  if (!h) return MOE_TAIL_ERR_INVALID_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e);
  int32_t v = 0;
  e = cudaMemcpy(&v, h->s.status, 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e);
  if (device_status) *device_status = v;
  if (v & kStatusTimeout) return MOE_TAIL_ERR_TIMEOUT;
  return v ? MOE_TAIL_ERR_DEVICE : MOE_TAIL_OK;
}

extern "C" int moe_tail_clear_status(moe_tail_t* h) {
  if (!h) return MOE_TAIL_ERR_INVALID_ARG;
  cudaError_t e = cudaMemset(h->s.status, 0, 4);
  // a persistent call that gave up may have left its barrier count behind
  if (e == cudaSuccess && h->cfg.mode == MOE_TAIL_MODE_PERSISTENT)
    e = persistent_reset(h->s);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  return e == cudaSuccess ? MOE_TAIL_OK : cuda_fail(e);
}

extern "C" int moe_tail_debug_routing(moe_tail_t* h, int32_t* ids, float* wts,
                                      int32_t* n_distinct, void* stream) {
  if (!h) return MOE_TAIL_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  const size_t P = (size_t)(h->last_rows > 0 ? h->last_rows : 0) * h->cfg.top_k;
  cudaError_t e = cudaSuccess;
  if (ids && P) e = cudaMemcpyAsync(ids, h->s.ids, P * 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess && wts && P) e = cudaMemcpyAsync(wts, h->s.wts, P * 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess && n_distinct)
    e = cudaMemcpyAsync(n_distinct, h->s.n_distinct, 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  return e == cudaSuccess ? MOE_TAIL_OK : cuda_fail(e);
}

extern "C" int moe_tail_debug_timeline(moe_tail_t* h, uint64_t* stamps, int32_t n) {
  if (!h || !stamps || n < 0) return MOE_TAIL_ERR_INVALID_ARG;
  if (!h->s.tl) return MOE_TAIL_ERR_UNSUPPORTED;
  cudaError_t e = cudaDeviceSynchronize();
  const int m = n < kTlSlots ? n : kTlSlots;
  if (e == cudaSuccess && m > 0)
    e = cudaMemcpy(stamps, h->s.tl, (size_t)m * 8, cudaMemcpyDeviceToHost);
  return e == cudaSuccess ? m : cuda_fail(e);
}

extern "C" void moe_tail_destroy(moe_tail_t* h) {
  if (!h) return;
  int cur = -1;
  cudaGetDevice(&cur);
  if (cur != h->device) cudaSetDevice(h->device);
  cudaDeviceSynchronize();
  cudaFree(h->slab);
  cudaFree(h->stage);
  if (h->atoms) cudaFree(h->atoms);
  for (int r = 0; r <= kMaxRows; ++r) {
    if (h->hexec[r]) cudaGraphExecDestroy(h->hexec[r]);
    if (h->hgraph[r]) cudaGraphDestroy(h->hgraph[r]);
  }
  if (h->hdone) cudaFreeHost(h->hdone);
  if (cur >= 0 && cur != h->device) cudaSetDevice(cur);
  delete h;
}

extern "C" int moe_tail_refresh_scales(moe_tail_t* h, void* stream) {
  if (!h) return MOE_TAIL_ERR_INVALID_ARG;
  if (!h->atoms) return MOE_TAIL_OK;  // a form that reads w13s and w2s in place
  Dims d0;
  d0.R = h->cfg.max_rows; d0.Rmax = h->cfg.max_rows; d0.H = h->cfg.hidden;
  d0.E = h->cfg.n_experts; d0.k = h->cfg.top_k; d0.I = h->cfg.expert_inter;
  d0.Is = h->cfg.shared_inter; d0.eps = h->cfg.rms_eps; d0.Ha = h->cfg.attn_dim; d0.Pk = 1;
  const cudaError_t e = launch_scale_atoms(d0, h->w, (uint8_t*)h->atoms, (cudaStream_t)stream);
  return e == cudaSuccess ? MOE_TAIL_OK : cuda_fail(e);
}

// ------------------------------------------- the AttnRes residual mix (attnres_mix.h) ----

extern "C" int moe_attnres_mix_ctas_per_row(int hidden, int n_blocks) {
  amix::MixPlan p;
  if (n_blocks < 0 || !amix::mix_plan(hidden, n_blocks + 1, &p)) return MOE_TAIL_ERR_UNSUPPORTED;
  return p.C;
}

extern "C" int moe_attnres_mix(int rows, int hidden, int n_blocks, int commit, float eps,
                               const void* sub, void* prefix, void* blocks, const void* q,
                               const void* gamma, void* mix, void* y, unsigned flags,
                               void* stream) {
  if (rows < 1 || rows > amix::kMaxRows || n_blocks < 0) return MOE_TAIL_ERR_INVALID_ARG;
  if (!(eps > 0.f) || !isfinite(eps)) return MOE_TAIL_ERR_INVALID_ARG;
  if (flags & ~(unsigned)(MOE_ATTNRES_MIX_PDL | MOE_ATTNRES_MIX_DEBUG_STALL))
    return MOE_TAIL_ERR_INVALID_ARG;
  const bool need_blocks = n_blocks > 0 || commit;
  const void* ptrs[] = {sub, prefix, q, gamma, mix, y, need_blocks ? blocks : sub};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return MOE_TAIL_ERR_INVALID_ARG;
  amix::MixPlan plan;
  if (!amix::mix_plan(hidden, n_blocks + 1, &plan)) return MOE_TAIL_ERR_UNSUPPORTED;
  amix::MixArgs a;
  a.sub = (const uint16_t*)sub;
  a.prefix = (uint16_t*)prefix;
  a.blocks = (uint16_t*)blocks;
  a.q = (const uint16_t*)q;
  a.gamma = (const uint16_t*)gamma;
  a.mix = (uint16_t*)mix;
  a.y = (uint16_t*)y;
  a.R = rows;
  a.H = hidden;
  a.n_blocks = n_blocks;
  a.commit = commit ? 1 : 0;
  a.eps = eps;
  a.debug_stall = (flags & MOE_ATTNRES_MIX_DEBUG_STALL) ? 1 : 0;
  const cudaError_t e = amix::launch_attnres_mix(a, plan, (cudaStream_t)stream,
                                                 (flags & MOE_ATTNRES_MIX_PDL) != 0);
  return e == cudaSuccess ? MOE_TAIL_OK : cuda_fail(e);
}

extern "C" int moe_attnres_mix_get_status(int* status, int clear) {
  if (!status) return MOE_TAIL_ERR_INVALID_ARG;
  int v = 0;
  const cudaError_t e = amix::mix_status(&v, clear != 0);
  if (e != cudaSuccess) return cuda_fail(e);
  *status = v;
  return v ? MOE_TAIL_ERR_DEVICE : MOE_TAIL_OK;
}

extern "C" int moe_tail_check_scratch(moe_tail_t* h) {
  if (!h) return MOE_TAIL_ERR_INVALID_ARG;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e);
  unsigned char buf[kCanaryBytes];
  for (int i = 0; i < h->n_canary; ++i) {
    e = cudaMemcpy(buf, (const char*)h->slab + h->canary_off[i], kCanaryBytes,
                   cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    for (size_t b = 0; b < kCanaryBytes; ++b)
      if (buf[b] != kCanaryByte) {
        snprintf(g_cuda_err, sizeof(g_cuda_err), "scratch guard %d overwritten at byte %zu", i,
                 b);
        return MOE_TAIL_ERR_DEVICE;
      }
  }
  return MOE_TAIL_OK;
}
