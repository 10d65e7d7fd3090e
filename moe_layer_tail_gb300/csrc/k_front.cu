// k_front.cu -- the front of the tail: residual add + RMSNorm, router GEMV, top-k and the
// expert dedup that builds the call's work list.
//
// Sources: "[AMD] integrate kimi k3 monokernel" page, Kernel Replacement table rows "The
// post-attention norm", "The router" and "The top-k"; "glm53: Long-context indexer ..."
// page, Modifications table rows 9 (ties run the id reduction only when the maximum is
// shared), 10 (bf16 activations before the router), 16 and 20 (each distinct expert once,
// users in row order), and its reviewer note that every CTA routes all rows, so no
// cross-CTA hand-off of the routing is needed.
//
// Two forms: k_front_fused (one launch: every CTA recomputes the row norms it needs, runs
// its slice of the router, and the last CTA to finish runs top-k and the dedup), and the
// three single-purpose kernels k_add_rmsnorm / k_router / k_topk_dedup used by the
// cross-checking path.  bf16(x + residual) goes to scratch; the residual itself is
// rewritten by the combine, after every reader is done.
#include <algorithm>
#include <cstddef>
#include <mutex>

#include "k_front.cuh"
#include "moe_tail.h"
#include "moe_tail_internal.cuh"

namespace mtail {

// ---------------------------------------------------------------- add + RMSNorm ----
// One CTA of 512 threads per row.  Thread i owns the 16-byte groups i, i + 512, ... of the
// row (up to 8, H <= 32768) and keeps bf16(x + residual) in registers; gamma is staged in
// shared memory before the wait on the previous launch (it depends on nothing).  Two block
// reductions (sum of squares, then max |n|) in a fixed order; no value is re-read from
// global memory.
constexpr int kNormThreads = 512;
constexpr int kNormGroups = 8;


__global__ void __launch_bounds__(kNormThreads)
k_add_rmsnorm(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ residual,
              const __nv_bfloat16* __restrict__ gamma, __nv_bfloat16* __restrict__ rnew,
              __nv_bfloat16* __restrict__ n_out, __half* __restrict__ n16,
              float* __restrict__ n16s, uint32_t* __restrict__ counters, int H, float eps,
              const __nv_bfloat16* __restrict__ wsg, float* __restrict__ sgate,
              const float* __restrict__ xpart, int Pk, size_t part_stride,
              uint8_t* __restrict__ np4, uint8_t* __restrict__ np4a,
              unsigned long long* __restrict__ tl, const HostArgs* ha) {
  extern __shared__ uint4 s_gamma[];  // [H / 8]
  __shared__ float part[kNormThreads / 32];
  const int r = blockIdx.x;
  // a host-buffer call: its buffers (written before the launch), read once per CTA, over the
  // link while gamma is staged
  const void* hx = nullptr;
  const void* hr = nullptr;
  if (ha && threadIdx.x == 0) {
    hx = ha_ptr(&ha->x);
    hr = ha_ptr((const void* const*)&ha->residual);
  }
  const uint4* g4 = reinterpret_cast<const uint4*>(gamma);
  for (int c = threadIdx.x; c < H / 8; c += kNormThreads) s_gamma[c] = __ldg(g4 + c);
  pdl_wait();
  pdl_trigger();
  if (ha) {
    __shared__ const void* s_buf[2];
    if (threadIdx.x == 0) {
      s_buf[0] = hx;
      s_buf[1] = hr;
    }
    __syncthreads();
    x = reinterpret_cast<const __nv_bfloat16*>(s_buf[0]);
    residual = reinterpret_cast<const __nv_bfloat16*>(s_buf[1]);
  }
  if (threadIdx.x == 0) tl_first(tl, kTlNormStart);
  if (r == 0)  // work counters, tickets and per-expert progress of this call
    for (int i = threadIdx.x; i < kCtrWords; i += kNormThreads) counters[i] = 0u;
  add_rmsnorm_row<kNormThreads, kNormGroups>(r, x, residual, s_gamma, rnew, n_out, n16, n16s, H,
                                             eps, wsg, sgate, xpart, Pk, part_stride, np4, np4a,
                                             part);
  if (tl) {
    __syncthreads();
    if (threadIdx.x == 0) tl_last(tl, kTlNormEnd);
  }
}

cudaError_t launch_add_rmsnorm(const Dims& d, const __nv_bfloat16* x,
                               const __nv_bfloat16* residual, const Weights& w,
                               const Scratch& s, cudaStream_t st, bool pdl, const float* xpart,
                               bool planes, const HostArgs* ha) {
  return launch_k(k_add_rmsnorm, dim3(d.R), dim3(kNormThreads), (size_t)d.H * 2, st, pdl, x,
                  residual, w.gamma, s.rnew, s.n, s.n16, s.n16s, s.counters, d.H, d.eps, w.wsg,
                  s.sgate, xpart, d.Pk, (size_t)d.Rmax * d.H, planes ? s.np4 : nullptr,
                  planes ? s.np4a : nullptr, s.tl, ha);
}

// ------------------------------------------------------------------- router GEMV ----
// One warp per expert: lanes stride over 8-element chunks of the router row and of every
// activation row; fp32 accumulation in a fixed order, butterfly reduction.
constexpr int kRouterWarps = 8;

__global__ void __launch_bounds__(kRouterWarps * 32)
k_router(const __nv_bfloat16* __restrict__ n, const __nv_bfloat16* __restrict__ w_r,
         float* __restrict__ logits, int R, int H, int E) {
  const int lane = threadIdx.x & 31;
  const int e = blockIdx.x * kRouterWarps + (threadIdx.x >> 5);
  pdl_wait();
  pdl_trigger();
  if (e >= E) return;
  router_warp(n, w_r, logits, R, H, E, e, lane);
}

cudaError_t launch_router(const Dims& d, const Weights& w, const Scratch& s, cudaStream_t st,
                          bool pdl) {
  dim3 grid((d.E + kRouterWarps - 1) / kRouterWarps);
  return launch_k(k_router, grid, dim3(kRouterWarps * 32), 0, st, pdl,
                  (const __nv_bfloat16*)s.n, w.w_r, s.logits, d.R, d.H, d.E);
}

// top-k + dedup: topk_dedup_block and its helpers are in k_front.cuh

constexpr int kTopkThreads = 512;

__global__ void __launch_bounds__(kTopkThreads)
k_topk_dedup(const float* __restrict__ logits, int32_t* __restrict__ ids,
             float* __restrict__ wts, int32_t* __restrict__ n_distinct,
             int32_t* __restrict__ uniq, int32_t* __restrict__ user_off,
             int32_t* __restrict__ user_list, int32_t* __restrict__ status, int R, int E,
             int k) {
  pdl_wait();
  pdl_trigger();
  topk_dedup_block<false>(logits, ids, wts, n_distinct, uniq, user_off, user_list, status, R, E,
                          k);
}

cudaError_t launch_topk_dedup(const Dims& d, const Scratch& s, cudaStream_t st, bool pdl) {
  return launch_k(k_topk_dedup, dim3(1), dim3(kTopkThreads), 0, st, pdl,
                  (const float*)s.logits, s.ids, s.wts, s.n_distinct, s.uniq, s.user_off,
                  s.user_list, s.status, d.R, d.E, d.k);
}

// --------------------------------------------------------------- router + top-k ----
// Grid (ceil(E / 16), P): CTA (x, p) computes the logits of experts 16x .. 16x+15 for every
// row over K part p of H, on the tensor cores (mma.m16n8k16, bf16 x bf16 into fp32; the 16
// experts are the M rows, the call's rows the N columns).  The CTA's router weights are
// copied into shared memory with cp.async before the wait on the norm launch (they depend
// on nothing), then the rows' n for the part (up to 32 rows: four N-tiles of 8); each of
// the 16 warps takes a slice of the part's 32-element K steps and the warps' partial tiles
// are added in warp order.  The
// partial logits of each part go to scratch; the last CTA to finish (atomic ticket after a
// fence) adds the parts in part order into shared memory, then runs top-k (one warp per row,
// so 16 warps take up to 16 rows at once: a row's selection is a chain of dependent warp
// reductions, ~1.5 us whatever else runs) and the dedup.
// Loops stay rolled: every CTA runs this code once, so its size, not its instruction
// count, sets the time an SM waits for instructions.
constexpr int kRtWarps = 16;
constexpr int kRtThreads = kRtWarps * 32;

// Parts: enough CTAs to spread the router weights over the SMs (about 128), parts of at
// most 2048 elements, each a multiple of 32; the shared memory of a part for `warps` warps
// (the largest of the staged weights and rows, the logits of the last part and the warps'
// tiles: each overlays the one before).
RouterPlan router_plan(int R, int H, int E, int warps) {
  RouterPlan p;
  p.tiles = (E + kRtTile - 1) / kRtTile;
  int P = (128 + p.tiles - 1) / p.tiles;
  P = std::max(P, (H + kRtMaxPart - 1) / kRtMaxPart);
  P = std::min(P, kRtMaxParts);
  const size_t nt = (R + 7) / 8;
  for (;; ++P) {  // more parts while the staged rows of many-row handles exceed 192 KB
    p.plen = ((H + P - 1) / P + 31) / 32 * 32;
    p.parts = (H + p.plen - 1) / p.plen;
    const size_t pitch = (size_t)p.plen * 2 + 16;
    const size_t tiles_bytes = (kRtTile + (size_t)R) * pitch;
    const size_t logit_bytes = (size_t)R * E * 4;
    // the warps' reduction tiles overlay the staged tiles once every warp's MMAs are done
    const size_t red_bytes = (size_t)warps * nt * 32 * 16;
    p.red_off = 0;
    p.smem = ((std::max(std::max(tiles_bytes, logit_bytes), red_bytes) + 15) / 16) * 16;
    if (p.smem <= 192 * 1024 || P >= kRtMaxParts) break;
  }
  return p;
}

// Grid (tiles, parts): one router part per CTA (router_stage_w before the wait on the norm
// launch, router_part after it); the last part runs router_finish.  Loops stay rolled: every
// CTA runs this code once, so its size, not its instruction count, sets the time an SM waits
// for instructions.
__global__ void __launch_bounds__(kRtThreads)
k_router_topk(const __nv_bfloat16* __restrict__ w_r, Scratch s, int R, int H, int E, int k,
              int plen, int red_off) {
  extern __shared__ __align__(16) uint8_t sm[];
  __shared__ int s_last;
  router_stage_w<kRtThreads>(sm, w_r, blockIdx.x, blockIdx.y, plen, H, E);
  pdl_wait();
  if (threadIdx.x == 0) {
    tl_first(s.tl, kTlRouterStart);
    tl_last(s.tl, kTlRouterAllStarted);
  }
  // the expert launch may start as soon as every router CTA is past its wait: its
  // shared-expert items need only n (written by the norm launch, complete by now), and its
  // routed items wait for the kCtrRouted word this launch's last CTA sets
  pdl_trigger();
  if (router_part<kRtWarps>(sm, s, blockIdx.x, blockIdx.y, plen, red_off, R, H, E,
                            gridDim.x * gridDim.y, &s_last))
    router_finish<kRtThreads, false>(sm, s, gridDim.y, R, E, k);
}

cudaError_t launch_router_topk(const Dims& d, const Weights& w, const Scratch& s,
                               cudaStream_t st, bool pdl) {
  const RouterPlan rp = router_plan(d.R, d.H, d.E, kRtWarps);
  return launch_k(k_router_topk, dim3(rp.tiles, rp.parts), dim3(kRtThreads), rp.smem, st, pdl,
                  w.w_r, s, d.R, d.H, d.E, d.k, rp.plen, rp.red_off);
}

// Parts of the router's K at most: sizes the scratch of the partial logits.
int router_max_parts() { return kRtMaxParts; }

// The norm kernel stages gamma (up to 64 KB) and the router kernel its weight tile and n
// (up to 2 x 16 rows of 2048 bf16 plus the reduction tiles) in dynamic shared memory.
cudaError_t prepare_front_kernels() {
  cudaError_t e = cudaFuncSetAttribute(k_add_rmsnorm, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (1 << 15) * 2);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_router_topk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)router_plan(kMaxRows, 1 << 15, kMaxExperts, kRtWarps).smem + 4096);
  return e;
}

// ------------------------------------------------------------------- fused front ----
// One launch of ceil(E / 8) CTAs x 8 warps.  Every CTA computes rstd of every row (same
// code and order in every CTA, so all agree bitwise), then walks H in chunks: the CTA
// builds n = bf16(bf16(x + res) * rstd * gamma) for the chunk in shared memory and its
// 8 warps (one expert each) accumulate their router dot products.  Chunk c's values are
// also stored to scratch (r_new, n, and n's f16 copy) by CTA c % grid only.  The last CTA
// to finish (atomic ticket after a fence) runs top-k and the dedup, and clears the
// counters of the expert launches.
constexpr int kFrontWarps = 8;
constexpr int kFrontThreads = kFrontWarps * 32;
constexpr int kFrontChunk = 1024;

__global__ void __launch_bounds__(kFrontThreads)
k_front_fused(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ residual,
              const __nv_bfloat16* __restrict__ gamma, const __nv_bfloat16* __restrict__ w_r,
              Scratch s, int R, int H, int E, int k, float eps) {
  __shared__ float s_rstd[kMaxRowsOther];
  __shared__ float s_down[kMaxRowsOther];
  __shared__ float s_gmax[kFrontWarps];
  __shared__ uint4 s_n[kMaxRowsOther][kFrontChunk / 8];
  __shared__ int s_last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x;
  pdl_wait();
  pdl_trigger();

  // 1. rstd of every row (warp w sums rows w, w + 8 in a fixed order), the row maxima of
  //    |r_new| and the maximum of |gamma|: their product bounds |n| and fixes the row's
  //    power-of-two scale for the f16 copy (row maximum below 2^15).
  const uint4* g4 = reinterpret_cast<const uint4*>(gamma);
  {
    float gm = 0.f;
#pragma unroll 4
    for (int c = tid; c < H / 8; c += kFrontThreads) gm = fmaxf(gm, group_amax(__ldg(g4 + c)));
    gm = warp_max(gm);
    if (lane == 0) s_gmax[warp] = gm;
  }
  __syncthreads();
  float gmax = 0.f;
  for (int i = 0; i < kFrontWarps; ++i) gmax = fmaxf(gmax, s_gmax[i]);
  for (int r = warp; r < R; r += kFrontWarps) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)r * H);
    const uint4* rr = reinterpret_cast<const uint4*>(residual + (size_t)r * H);
    float ss = 0.f, rmax = 0.f;
#pragma unroll 4
    for (int c = lane; c < H / 8; c += 32) {
      const uint4 xv = __ldg(xr + c), rv = __ldg(rr + c);
      const uint4 o4 = make_uint4(add_bf16x2(xv.x, rv.x), add_bf16x2(xv.y, rv.y),
                                  add_bf16x2(xv.z, rv.z), add_bf16x2(xv.w, rv.w));
      const uint32_t o[4] = {o4.x, o4.y, o4.z, o4.w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        ss += bf16_lo(o[q]) * bf16_lo(o[q]) + bf16_hi(o[q]) * bf16_hi(o[q]);
      rmax = fmaxf(rmax, group_amax(o4));
    }
    ss = warp_sum(ss);
    rmax = warp_max(rmax);
    const float rstd = 1.0f / sqrtf(ss / (float)H + eps);
    const int p = f16_block_exp(rmax * rstd * gmax * 1.0078125f);
    if (lane == 0) {
      s_rstd[r] = rstd;
      s_down[r] = __uint_as_float((uint32_t)(127 - p) << 23);
      if (blockIdx.x == 0) s.n16s[r] = __uint_as_float((uint32_t)(127 + p) << 23);
    }
  }
  __syncthreads();

  // 2. router over H in chunks
  const int e = blockIdx.x * kFrontWarps + warp;
  float acc[kMaxRowsOther];
#pragma unroll
  for (int r = 0; r < kMaxRowsOther; ++r) acc[r] = 0.f;
  for (int h0 = 0, ci = 0; h0 < H; h0 += kFrontChunk, ++ci) {
    const int cw = min(kFrontChunk, H - h0);  // multiple of 128
    const int ng = cw / 8;                     // 16-byte groups per row in this chunk
    const bool owner = (ci % G) == (int)blockIdx.x;
    // this warp's router weights for the chunk, loaded before n is built (up to 4 groups
    // of 8 per lane: kFrontChunk / 8 / 32)
    uint4 wreg[kFrontChunk / 8 / 32];
#pragma unroll
    for (int q = 0; q < kFrontChunk / 8 / 32; ++q) {
      const int c = lane + 32 * q;
      wreg[q] = (e < E && c < ng)
                    ? __ldg(reinterpret_cast<const uint4*>(w_r + (size_t)e * H + h0) + c)
                    : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll 4
    for (int idx = tid; idx < R * ng; idx += kFrontThreads) {
      const int r = idx / ng, gidx = idx % ng;
      const size_t off = ((size_t)r * H + h0) / 8 + gidx;
      const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x) + off);
      const uint4 rv = __ldg(reinterpret_cast<const uint4*>(residual) + off);
      const uint4 gv = __ldg(g4 + h0 / 8 + gidx);
      const uint4 rn = make_uint4(add_bf16x2(xv.x, rv.x), add_bf16x2(xv.y, rv.y),
                                  add_bf16x2(xv.z, rv.z), add_bf16x2(xv.w, rv.w));
      const float rs = s_rstd[r];
      const uint4 nv = make_uint4(norm_bf16x2(rn.x, gv.x, rs), norm_bf16x2(rn.y, gv.y, rs),
                                  norm_bf16x2(rn.z, gv.z, rs), norm_bf16x2(rn.w, gv.w, rs));
      s_n[r][gidx] = nv;
      if (owner) {
        reinterpret_cast<uint4*>(s.rnew)[off] = rn;
        reinterpret_cast<uint4*>(s.n)[off] = nv;
        reinterpret_cast<uint4*>(s.n16)[off] = f16_group(nv, s_down[r]);
      }
    }
    __syncthreads();
    if (e < E) {
#pragma unroll
      for (int q = 0; q < kFrontChunk / 8 / 32; ++q) {
        const int c = lane + 32 * q;
        if (c >= ng) break;
        const uint4 wv = wreg[q];
        const float wf[8] = {bf16_lo(wv.x), bf16_hi(wv.x), bf16_lo(wv.y), bf16_hi(wv.y),
                             bf16_lo(wv.z), bf16_hi(wv.z), bf16_lo(wv.w), bf16_hi(wv.w)};
#pragma unroll
        for (int r = 0; r < kMaxRowsOther; ++r) {
          if (r < R) {
            const uint4 nv = s_n[r][c];
            float a = acc[r];
            a += wf[0] * bf16_lo(nv.x); a += wf[1] * bf16_hi(nv.x);
            a += wf[2] * bf16_lo(nv.y); a += wf[3] * bf16_hi(nv.y);
            a += wf[4] * bf16_lo(nv.z); a += wf[5] * bf16_hi(nv.z);
            a += wf[6] * bf16_lo(nv.w); a += wf[7] * bf16_hi(nv.w);
            acc[r] = a;
          }
        }
      }
    }
    __syncthreads();
  }
  if (e < E) {
#pragma unroll
    for (int r = 0; r < kMaxRowsOther; ++r) {
      if (r < R) {
        const float v = warp_sum(acc[r]);
        if (lane == 0) s.logits[(size_t)r * E + e] = v;
      }
    }
  }

  // 3. the last CTA to finish ranks the experts and builds the work list
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const uint32_t t = atomicAdd(&s.counters[kCtrFrontTicket], 1u);
    s_last = (t == (uint32_t)(G - 1)) ? 1 : 0;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  topk_dedup_block<false>(s.logits, s.ids, s.wts, s.n_distinct, s.uniq, s.user_off,
                          s.user_list, s.status, R, E, k);
  // the ticket and the expert launch's counters for this call (every other CTA is done)
  for (int i = tid; i < kCtrWords; i += kFrontThreads) s.counters[i] = 0u;
}

cudaError_t launch_front_fused(const Dims& d, const __nv_bfloat16* x,
                               const __nv_bfloat16* residual, const Weights& w,
                               const Scratch& s, cudaStream_t st, bool pdl) {
  dim3 grid((d.E + kFrontWarps - 1) / kFrontWarps);
  return launch_k(k_front_fused, grid, dim3(kFrontThreads), 0, st, pdl, x, residual, w.gamma,
                  w.w_r, s, d.R, d.H, d.E, d.k, d.eps);
}

}  // namespace mtail

// ------------------------------------------- routing without any allocation ----
// The routing of one call (add + RMSNorm, router GEMV, top-k with renormalised weights)
// for callers that cannot allocate device memory: everything the launch needs besides its
// inputs and outputs lives in the file-scope array below, which every GPU that loads this
// library holds until the process exits.  Its size bounds the call: rows <= 16 and
// n_experts <= 1024 (the fp32 logits), plus the dedup tables and the ticket counter.

namespace mtail {

struct RouteScratch {
  float logits[kMaxRowsOther * kMaxExperts];
  int32_t n_distinct;
  int32_t uniq[kMaxRowsOther * kMaxTopK];
  int32_t user_off[kMaxRowsOther * kMaxTopK + 1];
  int32_t user_list[kMaxRowsOther * kMaxTopK];
  int32_t status;   // status bits of the running call (cleared with the ticket)
  uint32_t ticket;  // CTAs done with their logits (the last one ranks)
};

static_assert(sizeof(RouteScratch) == 71696, "the size stated in moe_tail.h");
static __device__ __align__(256) uint8_t g_route_scratch[sizeof(RouteScratch)];

// Same arithmetic as k_front_fused, the fused-front form of moe_tail_run (same rstd, n
// and logit order, same top-k), without the stores the expert stages need; ids, wts,
// n_distinct and the call's status bits go to the caller's buffers.
__global__ void __launch_bounds__(kFrontThreads)
k_route_static(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ residual,
               const __nv_bfloat16* __restrict__ gamma, const __nv_bfloat16* __restrict__ w_r,
               RouteScratch* __restrict__ rs, int32_t* __restrict__ ids_out,
               float* __restrict__ wts_out, int32_t* __restrict__ nd_out,
               int32_t* __restrict__ status_out, int R, int H, int E, int k, float eps) {
  __shared__ float s_rstd[kMaxRowsOther];
  __shared__ uint4 s_n[kMaxRowsOther][kFrontChunk / 8];
  __shared__ int s_last;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x;
  const uint4* g4 = reinterpret_cast<const uint4*>(gamma);
  for (int r = warp; r < R; r += kFrontWarps) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)r * H);
    const uint4* rr = reinterpret_cast<const uint4*>(residual + (size_t)r * H);
    float ss = 0.f;
#pragma unroll 4
    for (int c = lane; c < H / 8; c += 32) {
      const uint4 xv = __ldg(xr + c), rv = __ldg(rr + c);
      const uint32_t o[4] = {add_bf16x2(xv.x, rv.x), add_bf16x2(xv.y, rv.y),
                             add_bf16x2(xv.z, rv.z), add_bf16x2(xv.w, rv.w)};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        ss += bf16_lo(o[q]) * bf16_lo(o[q]) + bf16_hi(o[q]) * bf16_hi(o[q]);
    }
    ss = warp_sum(ss);
    if (lane == 0) s_rstd[r] = 1.0f / sqrtf(ss / (float)H + eps);
  }
  __syncthreads();
  const int e = blockIdx.x * kFrontWarps + warp;
  float acc[kMaxRowsOther];
#pragma unroll
  for (int r = 0; r < kMaxRowsOther; ++r) acc[r] = 0.f;
  for (int h0 = 0; h0 < H; h0 += kFrontChunk) {
    const int ng = min(kFrontChunk, H - h0) / 8;
    for (int idx = tid; idx < R * ng; idx += kFrontThreads) {
      const int r = idx / ng, gidx = idx % ng;
      const size_t off = ((size_t)r * H + h0) / 8 + gidx;
      const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x) + off);
      const uint4 rv = __ldg(reinterpret_cast<const uint4*>(residual) + off);
      const uint4 gv = __ldg(g4 + h0 / 8 + gidx);
      const uint4 rn = make_uint4(add_bf16x2(xv.x, rv.x), add_bf16x2(xv.y, rv.y),
                                  add_bf16x2(xv.z, rv.z), add_bf16x2(xv.w, rv.w));
      const float rsd = s_rstd[r];
      s_n[r][gidx] = make_uint4(norm_bf16x2(rn.x, gv.x, rsd), norm_bf16x2(rn.y, gv.y, rsd),
                                norm_bf16x2(rn.z, gv.z, rsd), norm_bf16x2(rn.w, gv.w, rsd));
    }
    __syncthreads();
    if (e < E) {
      const uint4* wrow = reinterpret_cast<const uint4*>(w_r + (size_t)e * H + h0);
      for (int c = lane; c < ng; c += 32) {
        const uint4 wv = __ldg(wrow + c);
        const float wf[8] = {bf16_lo(wv.x), bf16_hi(wv.x), bf16_lo(wv.y), bf16_hi(wv.y),
                             bf16_lo(wv.z), bf16_hi(wv.z), bf16_lo(wv.w), bf16_hi(wv.w)};
#pragma unroll
        for (int r = 0; r < kMaxRowsOther; ++r) {
          if (r < R) {
            const uint4 nv = s_n[r][c];
            float a = acc[r];
            a += wf[0] * bf16_lo(nv.x); a += wf[1] * bf16_hi(nv.x);
            a += wf[2] * bf16_lo(nv.y); a += wf[3] * bf16_hi(nv.y);
            a += wf[4] * bf16_lo(nv.z); a += wf[5] * bf16_hi(nv.z);
            a += wf[6] * bf16_lo(nv.w); a += wf[7] * bf16_hi(nv.w);
            acc[r] = a;
          }
        }
      }
    }
    __syncthreads();
  }
  if (e < E) {
#pragma unroll
    for (int r = 0; r < kMaxRowsOther; ++r) {
      if (r < R) {
        const float v = warp_sum(acc[r]);
        if (lane == 0) rs->logits[(size_t)r * E + e] = v;
      }
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(&rs->ticket, 1u) == (uint32_t)(G - 1)) ? 1 : 0;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  topk_dedup_block<false>(rs->logits, ids_out, wts_out, &rs->n_distinct, rs->uniq, rs->user_off,
                   rs->user_list, &rs->status, R, E, k);
  __syncthreads();
  if (tid == 0) {
    if (nd_out) *nd_out = rs->n_distinct;
    if (status_out) *status_out = *(volatile int32_t*)&rs->status;
    rs->ticket = 0u;
  }
}

// Device address of the scratch array, looked up once per device (with that device
// current) the first time the entry point runs on it; std::call_once makes the lookup
// and its publication safe when several host threads make that first call together.
constexpr int kRouteMaxDevices = 64;
static std::once_flag g_route_once[kRouteMaxDevices];
static void* g_route_scratch_ptr[kRouteMaxDevices];
static cudaError_t g_route_scratch_err[kRouteMaxDevices];

}  // namespace mtail

extern "C" int moe_tail_route_noalloc(const void* x, const void* residual, const void* gamma,
                                      const void* router_w, int32_t rows, int32_t hidden,
                                      int32_t n_experts, int32_t top_k, float rms_eps,
                                      int32_t* ids, float* wts, int32_t* n_distinct,
                                      int32_t* status, void* stream) {
  using namespace mtail;
  if (!x || !residual || !gamma || !router_w || !ids || !wts) return MOE_TAIL_ERR_INVALID_ARG;
  const void* ptrs[4] = {x, residual, gamma, router_w};
  for (const void* p : ptrs)
    if ((uintptr_t)p & 15u) return MOE_TAIL_ERR_INVALID_ARG;
  if (rows < 1 || rows > kMaxRowsOther || n_experts < 1 || n_experts > kMaxExperts || top_k < 1 ||
      top_k > kMaxTopK || top_k > n_experts || hidden < 128 || hidden % 128 != 0 ||
      !(rms_eps > 0.f))
    return MOE_TAIL_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kRouteMaxDevices)
    return MOE_TAIL_ERR_CUDA;
  std::call_once(g_route_once[dev], [dev]() {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e == cudaSuccess && p == nullptr) e = cudaErrorInvalidSymbol;
    g_route_scratch_err[dev] = e;
    g_route_scratch_ptr[dev] = (e == cudaSuccess) ? p : nullptr;
  });
  if (g_route_scratch_err[dev] != cudaSuccess) return MOE_TAIL_ERR_CUDA;
  RouteScratch* rs = (RouteScratch*)g_route_scratch_ptr[dev];
  cudaStream_t st = (cudaStream_t)stream;
  // the status word and the ticket must start at zero (the status word holds the previous
  // call's bits; a call that stopped part-way could have left the ticket set); they are
  // adjacent in the array, so one memset clears both
  static_assert(offsetof(RouteScratch, ticket) == offsetof(RouteScratch, status) + 4,
                "status and ticket adjacent");
  if (cudaMemsetAsync(&rs->status, 0, 8, st) != cudaSuccess) return MOE_TAIL_ERR_CUDA;
  const int grid = (n_experts + kFrontWarps - 1) / kFrontWarps;
  k_route_static<<<grid, kFrontThreads, 0, st>>>(
      (const __nv_bfloat16*)x, (const __nv_bfloat16*)residual, (const __nv_bfloat16*)gamma,
      (const __nv_bfloat16*)router_w, rs, ids, wts, n_distinct, status, rows, hidden, n_experts,
      top_k, rms_eps);
  return cudaGetLastError() == cudaSuccess ? MOE_TAIL_OK : MOE_TAIL_ERR_CUDA;
}
