// k_mix.cu -- the AttnRes residual mix + RMSNorm of decode rows, one thread-block cluster
// per row.
//
// What one call computes ("Split the Kimi3 AttnRes mix across CTAs for decode rows",
// voipmonitor/flare #11, Description and commit message; the formulas are this library's
// reading, stated in attnres_mix.h): the residual add of the sublayer output into the
// block's running sum, the commit of a finished block, the softmax mixture of the row's
// sources (the committed blocks and the running sum) by query scores over RMS-normalised
// sources, and the RMSNorm of the bf16 mixture.
//
// The page splits a row over CTAs that exchange fp32 partials through global memory as
// (value, call tag) words and spin until the row's other CTAs have published, with a
// per-row epoch so that nothing is reset between calls.  Here the CTAs of a row form one
// thread-block cluster: the hardware schedules them together, each CTA stores its
// partials into a slot of every CTA's shared memory (distributed shared memory), and the
// receivers' mbarriers count the bytes in, which replaces the tagged words, the spins on
// global memory and the epochs (an mbarrier is initialised afresh by every launch).  As on the page,
// every CTA adds the partials in the same fixed order (its threads, then warps, then
// cluster ranks), so all CTAs of a row use bit-identical scores and norms.
//
// Two forms: k_attnres_mix_reg (chunks of at most 2048 columns, one thread per 16-byte vector,
// every source in registers; H 7168 and most shapes) and k_attnres_mix below (wider
// chunks, operands staged in shared memory, threads looping over several vectors).  With one
// vector per thread the two add in the same order.
//
// Per CTA (row r = blockIdx.y, chunk c = cluster rank, W columns):
//   1. cp.async stages the chunk of every source, the prefix, the sublayer output, q and
//      gamma in shared memory (each thread copies exactly the 16-byte vectors it later
//      uses, so no CTA barrier is needed before the arithmetic); q and gamma, which the
//      previous kernel does not write, are fetched before waiting for it, the rest is
//      prefetched into L2 before the wait and copied after it;
//   2. prefix' = bf16(prefix + sub), kept in shared memory as the last source;
//   3. per source: sum of squares and dot with q over the chunk, eight sources (sixteen
//      values) at a time reduced over the warp by a reduce-scatter butterfly (16 shuffles
//      instead of 80, the same addition tree as a full butterfly), added over warps;
//   4. the CTA's partials go to slot c of every CTA by asynchronous remote stores that
//      complete a transaction on the receiver's mbarrier; once all ranks' values are in,
//      each warp adds the slots in rank order and forms the scores and their softmax;
//   5. mixture h = bf16(sum_i alpha_i v_i) in source order (fp32 FMAs), stored; its
//      sum of squares travels the same way to a second mbarrier;
//   6. y = bf16(h * rstd * gamma); prefix (or the new block and a zero prefix) stored.
// One cluster barrier, arrived at the start and waited on before the first remote store,
// makes sure every CTA of the cluster is running (its mbarriers initialised) before another
// writes into its shared memory; once a CTA's second mbarrier has completed nothing writes
// into it any more, so each CTA exits as soon as it is done.  The mbarrier waits are
// bounded (50 ms); on expiry the device status word reports MOE_TAIL_STATUS_TIMEOUT.
#include <cuda_bf16.h>
#include <math.h>

#include <atomic>

#include "k_mix.cuh"
#include "moe_tail.h"
#include "moe_tail_internal.cuh"

namespace amix {

// The device's status word of the mix (MOE_TAIL_STATUS_* bits; moe_attnres_mix_get_status).
__device__ int g_mix_status;
constexpr uint64_t kWaitBudgetNs = 50ull * 1000 * 1000;

using mtail::bf16_hi;
using mtail::bf16_lo;
using mtail::pdl_trigger;
using mtail::pdl_wait;
using mtail::warp_max;
using mtail::warp_sum;

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
// Asynchronous store of a float into CTA `rank`'s shared memory at the address of `p` in
// this CTA's; its bytes count towards the transaction of that CTA's mbarrier `bar`.
__device__ __forceinline__ void st_async(float* p, uint32_t rank, float v, uint64_t* bar) {
  uint32_t ra, rb;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_u32(p)), "r"(rank));
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(smem_u32(bar)), "r"(rank));
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(ra),
               "r"(__float_as_uint(v)), "r"(rb)
               : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], 0;"
      " selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(b))
      : "memory");
  return ok != 0;
}
// Wait for the first phase of `b`, at most kWaitBudgetNs; on expiry the status word gets
// MOE_TAIL_STATUS_TIMEOUT and the caller goes on with whatever has arrived.
__device__ __forceinline__ void mbar_wait_bounded(uint64_t* b) {
  if (mbar_try(b)) return;
  const uint64_t t0 = mtail::globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try(b)) return;
    if ((i & 15) == 0 && mtail::globaltimer() - t0 > kWaitBudgetNs) {
      atomicOr(&g_mix_status, (int)MOE_TAIL_STATUS_TIMEOUT);
      return;
    }
  }
}
__device__ __forceinline__ void prefetch_l2(const void* g) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(g));
}
__device__ __forceinline__ void cp_async16(void* s, const void* g) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(s);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(a), "l"(g) : "memory");
}

__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
  f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x); f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
  f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z); f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
}
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);  // round to nearest even
  return *reinterpret_cast<const uint32_t*>(&b);
}
__device__ __forceinline__ uint4 pack8(const float* f) {
  return make_uint4(pack2(f[0], f[1]), pack2(f[2], f[3]), pack2(f[4], f[5]), pack2(f[6], f[7]));
}

__global__ void __launch_bounds__(kMaxThreads)
k_attnres_mix(const __grid_constant__ MixArgs a, int W, int C) {
  extern __shared__ uint4 sm[];
  __shared__ float red[kMaxThreads / 32][2 * kMaxSources];
  __shared__ float part1[kMaxCluster][2 * kMaxSources];  // [rank][2 i + (0: v.v, 1: q.v)]
  __shared__ float alpha_w[kMaxThreads / 32][kMaxSources];  // each warp's copy of alpha
  __shared__ float red2[kMaxThreads / 32];
  __shared__ float part2[kMaxCluster];                   // [rank] mixture square sums
  __shared__ __align__(8) uint64_t mbar[2];               // the two exchange rounds

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = blockDim.x, nwarps = T >> 5;
  const int r = blockIdx.y;
  const uint32_t c = cluster_rank();
  const int S = a.n_blocks + 1;
  const int nv = W >> 3;
  const float invH = 1.0f / (float)a.H;
  uint4* src = sm;                  // [S][nv]; source S - 1 is prefix'
  uint4* qv = sm + (size_t)S * nv;  // [nv]
  uint4* gv = qv + nv;              // [nv]
  uint4* pv = gv + nv;              // [nv] prefix as read, later the mixture h
  uint4* ov = pv + nv;              // [nv] sublayer output

  const size_t col0 = (size_t)c * W;
  const size_t row_off = (size_t)r * a.H + col0;
  const size_t blk_stride = (size_t)a.R * a.H;

  // The two exchange rounds land in this CTA's mbarriers, each expecting one fp32 value per
  // rank and entry (2S entries, then 1).  Every CTA of the cluster must be running, with its
  // mbarriers initialised, before another stores into its shared memory: arrive here, wait
  // before the first remote store.
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&mbar[0])));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&mbar[1])));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // the stall switch makes one CTA wait for a value that never comes (failure test)
    const uint32_t extra = (a.debug_stall && r == 0 && c == 0) ? 4u : 0u;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(&mbar[0])),
                 "r"((uint32_t)(C * 2 * S * 4))
                 : "memory");
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(&mbar[1])),
                 "r"((uint32_t)(C * 4) + extra)
                 : "memory");
  }
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");

  // 1. stage the chunk, each thread its own 16-byte vectors.  q and gamma are weights that
  //    the previous kernel does not write, so they are fetched before waiting for it; the
  //    rest is only prefetched into L2 (the point of coherence: a line fetched there early
  //    cannot be stale when it is read after the wait) and copied after the wait.
  for (int v = tid; v < nv; v += T) {
    cp_async16(&qv[v], a.q + col0 + 8 * v);
    cp_async16(&gv[v], a.gamma + col0 + 8 * v);
    for (int i = 0; i < a.n_blocks; ++i)
      prefetch_l2(a.blocks + i * blk_stride + row_off + 8 * v);
    prefetch_l2(a.prefix + row_off + 8 * v);
    prefetch_l2(a.sub + row_off + 8 * v);
  }
  pdl_wait();
  pdl_trigger();
  for (int v = tid; v < nv; v += T) {
    for (int i = 0; i < a.n_blocks; ++i)
      cp_async16(&src[(size_t)i * nv + v], a.blocks + i * blk_stride + row_off + 8 * v);
    cp_async16(&pv[v], a.prefix + row_off + 8 * v);
    cp_async16(&ov[v], a.sub + row_off + 8 * v);
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  asm volatile("cp.async.wait_group 0;" ::: "memory");

  // 2. residual add (the fp32 sum of two bf16 values rounds to the same bf16 as the exact
  //    sum: it is exact unless the exponents differ by more than 15, and then the smaller
  //    term is far below half a bf16 step of the larger)
  for (int v = tid; v < nv; v += T) {
    float p[8], o[8];
    unpack8(pv[v], p);
    unpack8(ov[v], o);
#pragma unroll
    for (int e = 0; e < 8; ++e) p[e] += o[e];
    src[(size_t)(S - 1) * nv + v] = pack8(p);
  }

  // 3. per-source partials, eight sources at a time: sum of squares and dot with q over
  //    this thread's vectors, then one reduce-scatter over the warp
  for (int i0 = 0; i0 < S; i0 += 8) {
    float ss[8], dt[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) ss[j] = dt[j] = 0.f;
    for (int v = tid; v < nv; v += T) {
      float qf[8];
      unpack8(qv[v], qf);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (i0 + j < S) {
          float x[8];
          unpack8(src[(size_t)(i0 + j) * nv + v], x);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            ss[j] = fmaf(x[e], x[e], ss[j]);
            dt[j] = fmaf(qf[e], x[e], dt[j]);
          }
        }
      }
    }
    // reduce-scatter butterfly: 16 values over 32 lanes in 8 + 4 + 2 + 1 + 1 shuffles;
    // lane L ends with value 8 b4 + 4 b3 + 2 b2 + b1 (b the bits of L)
    float vv[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) { vv[j] = ss[j]; vv[8 + j] = dt[j]; }
#pragma unroll
    for (int h = 8, o = 16; h >= 1; h >>= 1, o >>= 1) {
      const bool b = (lane & o) != 0;
#pragma unroll
      for (int k = 0; k < h; ++k) {
        const float send = b ? vv[k] : vv[k + h];
        const float keep = b ? vv[k + h] : vv[k];
        vv[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
      }
    }
    vv[0] += __shfl_xor_sync(0xffffffffu, vv[0], 1);
    {
      const int idx = ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 +
                      ((lane >> 1) & 1);
      const int j = idx & 7;
      if ((lane & 1) == 0 && i0 + j < S) red[warp][2 * (i0 + j) + (idx >> 3)] = vv[0];
    }
  }
  __syncthreads();

  // 4. this CTA's partials (warps in order) into slot c of every CTA of the row; after the
  //    barrier each CTA adds the slots in rank order
  cluster_wait();
  if (tid < 2 * S) {
    float s = 0.f;
    for (int w = 0; w < nwarps; ++w) s += red[w][tid];
    for (int k = 0; k < C; ++k) st_async(&part1[c][tid], (uint32_t)k, s, &mbar[0]);
  }
  mbar_wait_bounded(&mbar[0]);
  {
    // the scores and their softmax, lane i for source i, the same in every warp and CTA
    float sc = -INFINITY;
    if (lane < S) {
      float ssum = 0.f, dsum = 0.f;
      for (int k = 0; k < C; ++k) {
        ssum += part1[k][2 * lane];
        dsum += part1[k][2 * lane + 1];
      }
      sc = dsum * rsqrtf(fmaf(ssum, invH, a.eps));
    }
    const float m = warp_max(sc);
    const float e = lane < S ? expf(sc - m) : 0.f;
    const float den = __shfl_sync(0xffffffffu, warp_sum(e), 0);
    if (lane < S) alpha_w[warp][lane] = e / den;
    __syncwarp();
  }

  // 5. the mixture, its sum of squares, and the prefix / commit stores
  float hss = 0.f;
  for (int v = tid; v < nv; v += T) {
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int i = 0; i < S; ++i) {
      const float al = alpha_w[warp][i];
      float x[8];
      unpack8(src[(size_t)i * nv + v], x);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = fmaf(al, x[e], acc[e]);
    }
    const uint4 h = pack8(acc);
    pv[v] = h;
    *reinterpret_cast<uint4*>(a.mix + row_off + 8 * v) = h;
    float hf[8];
    unpack8(h, hf);
#pragma unroll
    for (int e = 0; e < 8; ++e) hss = fmaf(hf[e], hf[e], hss);
    const uint4 pn = src[(size_t)(S - 1) * nv + v];
    if (a.commit) {
      *reinterpret_cast<uint4*>(a.blocks + a.n_blocks * blk_stride + row_off + 8 * v) = pn;
      *reinterpret_cast<uint4*>(a.prefix + row_off + 8 * v) = make_uint4(0u, 0u, 0u, 0u);
    } else {
      *reinterpret_cast<uint4*>(a.prefix + row_off + 8 * v) = pn;
    }
  }
  hss = warp_sum(hss);
  if (lane == 0) red2[warp] = hss;
  __syncthreads();
  if (tid < C) {  // thread k sends this CTA's sum to rank k
    float s = 0.f;
    for (int w = 0; w < nwarps; ++w) s += red2[w];
    st_async(&part2[c], (uint32_t)tid, s, &mbar[1]);
  }
  // once every rank's value has landed no CTA writes into this one any more
  mbar_wait_bounded(&mbar[1]);

  // 6. the RMSNorm of the mixture
  float tot = 0.f;
  for (int k = 0; k < C; ++k) tot += part2[k];
  const float rs = rsqrtf(fmaf(tot, invH, a.eps));
  for (int v = tid; v < nv; v += T) {
    float hf[8], g[8];
    unpack8(pv[v], hf);
    unpack8(gv[v], g);
#pragma unroll
    for (int e = 0; e < 8; ++e) hf[e] = hf[e] * rs * g[e];
    *reinterpret_cast<uint4*>(a.y + row_off + 8 * v) = pack8(hf);
  }
}


// One level of the reduce-scatter butterfly: 2 HH values per lane become HH, summed with the
// lane O apart (the lane with bit O set keeps the upper half).
template <int HH, int O>
__device__ __forceinline__ void rs_level(float* vv, int lane) {
  const bool b = (lane & O) != 0;
#pragma unroll
  for (int k = 0; k < HH; ++k) {
    const float send = b ? vv[k] : vv[k + HH];
    const float keep = b ? vv[k + HH] : vv[k];
    vv[k] = keep + __shfl_xor_sync(0xffffffffu, send, O);
  }
}

// Source i of a thread: block i from the registers, prefix' at i == nb (selected by value, so
// that the register array is never indexed at run time).
template <int SMAX>
__device__ __forceinline__ uint4 source(const uint4 (&xs)[SMAX], int i, int nb, uint4 pn) {
  const uint4 b = xs[i];
  const bool p = (i == nb);
  return make_uint4(p ? pn.x : b.x, p ? pn.y : b.y, p ? pn.z : b.z, p ? pn.w : b.w);
}

// Square sums and q dots of sources I0 .. I0 + 7 (zero beyond the row's sources), reduced
// over the warp; the even lanes store the 16 totals into red_row.
template <int SMAX, int I0>
__device__ __forceinline__ void partials_group(const uint4 (&xs)[SMAX], uint4 pn, int nb,
                                               const float* qf, int S, int lane,
                                               float* red_row) {
  float vv[16];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float x[8];
    unpack8(source(xs, I0 + j, nb, pn), x);
    float ss = 0.f, dt = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      ss = fmaf(x[e], x[e], ss);
      dt = fmaf(qf[e], x[e], dt);
    }
    vv[j] = ss;
    vv[8 + j] = dt;
  }
  rs_level<8, 16>(vv, lane);
  rs_level<4, 8>(vv, lane);
  rs_level<2, 4>(vv, lane);
  rs_level<1, 2>(vv, lane);
  vv[0] += __shfl_xor_sync(0xffffffffu, vv[0], 1);
  const int idx = ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 +
                  ((lane >> 1) & 1);
  const int j = idx & 7;
  if ((lane & 1) == 0 && I0 + j < S) red_row[2 * (I0 + j) + (idx >> 3)] = vv[0];
}

// The same computation with every operand in registers, for chunks of at most 256 vectors
// (W <= 2048): one thread per 16-byte vector, up to SMAX sources held as uint4 registers.
// The loads go straight to registers (no shared-memory staging and no copy wait beyond the
// loads themselves), and both passes over the sources read registers.  Sources keep the
// order of the staged kernel (blocks, then prefix').
constexpr int kRegThreads = 256;

template <int SMAX>
__global__ void __launch_bounds__(kRegThreads)
k_attnres_mix_reg(const __grid_constant__ MixArgs a, int W, int C) {
  __shared__ float red[kRegThreads / 32][2 * SMAX];
  __shared__ float part1[kMaxCluster][2 * SMAX];        // [rank][2 i + (0: v.v, 1: q.v)]
  __shared__ float alpha_w[kRegThreads / 32][SMAX];     // each warp's copy of alpha
  __shared__ float red2[kRegThreads / 32];
  __shared__ float part2[kMaxCluster];                  // [rank] mixture square sums
  __shared__ __align__(8) uint64_t mbar[2];             // the two exchange rounds

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int r = blockIdx.y;
  const uint32_t c = cluster_rank();
  const int S = a.n_blocks + 1;
  const int nv = W >> 3;
  const int v = tid;
  const bool own = v < nv;
  const float invH = 1.0f / (float)a.H;
  const size_t col0 = (size_t)c * W;
  const size_t row_off = (size_t)r * a.H + col0 + 8 * (size_t)v;
  const size_t blk_stride = (size_t)a.R * a.H;

  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&mbar[0])));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&mbar[1])));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    const uint32_t extra = (a.debug_stall && r == 0 && c == 0) ? 4u : 0u;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(&mbar[0])),
                 "r"((uint32_t)(C * 2 * S * 4))
                 : "memory");
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_u32(&mbar[1])),
                 "r"((uint32_t)(C * 4) + extra)
                 : "memory");
  }
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");

  // 1. q and gamma (weights the previous kernel does not write) before the wait; the rest
  //    prefetched into L2 before it and loaded after it
  uint4 qv4 = make_uint4(0u, 0u, 0u, 0u), gv4 = qv4, pv4 = qv4, ov4 = qv4;
  uint4 xs[SMAX];
#pragma unroll
  for (int i = 0; i < SMAX; ++i) xs[i] = qv4;
  if (own) {
    qv4 = __ldg(reinterpret_cast<const uint4*>(a.q + col0) + v);
    gv4 = __ldg(reinterpret_cast<const uint4*>(a.gamma + col0) + v);
    for (int i = 0; i < a.n_blocks; ++i) prefetch_l2(a.blocks + i * blk_stride + row_off);
    prefetch_l2(a.prefix + row_off);
    prefetch_l2(a.sub + row_off);
  }
  pdl_wait();
  pdl_trigger();
  if (own) {
#pragma unroll
    for (int i = 0; i < SMAX - 1; ++i)
      if (i < a.n_blocks)
        xs[i] = *reinterpret_cast<const uint4*>(a.blocks + i * blk_stride + row_off);
    pv4 = *reinterpret_cast<const uint4*>(a.prefix + row_off);
    ov4 = *reinterpret_cast<const uint4*>(a.sub + row_off);
  }
  // 2. residual add (exact, as in the staged kernel); prefix' becomes source S - 1
  uint4 pn;
  {
    float p[8], o[8];
    unpack8(pv4, p);
    unpack8(ov4, o);
#pragma unroll
    for (int e = 0; e < 8; ++e) p[e] += o[e];
    pn = pack8(p);
  }

  // 3. per-source partials, eight sources at a time, reduce-scatter over the warp
  {
    float qf[8];
    unpack8(qv4, qf);
    partials_group<SMAX, 0>(xs, pn, a.n_blocks, qf, S, lane, red[warp]);
    if constexpr (SMAX > 8) {
      if (8 < S) partials_group<SMAX, 8>(xs, pn, a.n_blocks, qf, S, lane, red[warp]);
    }
    if constexpr (SMAX > 16) {
      if (16 < S) partials_group<SMAX, 16>(xs, pn, a.n_blocks, qf, S, lane, red[warp]);
      if (24 < S) partials_group<SMAX, 24>(xs, pn, a.n_blocks, qf, S, lane, red[warp]);
    }
  }
  __syncthreads();

  // 4. the exchange of the partials and the softmax, as in the staged kernel
  cluster_wait();
  if (tid < 2 * S) {
    float sum = 0.f;
    for (int w = 0; w < nwarps; ++w) sum += red[w][tid];
    for (int k = 0; k < C; ++k) st_async(&part1[c][tid], (uint32_t)k, sum, &mbar[0]);
  }
  mbar_wait_bounded(&mbar[0]);
  {
    float sc = -INFINITY;
    if (lane < S) {
      float ssum = 0.f, dsum = 0.f;
      for (int k = 0; k < C; ++k) {
        ssum += part1[k][2 * lane];
        dsum += part1[k][2 * lane + 1];
      }
      sc = dsum * rsqrtf(fmaf(ssum, invH, a.eps));
    }
    const float m = warp_max(sc);
    const float e = lane < S ? expf(sc - m) : 0.f;
    const float den = __shfl_sync(0xffffffffu, warp_sum(e), 0);
    if (lane < S) alpha_w[warp][lane] = e / den;
    __syncwarp();
  }

  // 5. the mixture from the registers, its sum of squares, the prefix / commit stores
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < SMAX; ++i) {
    if (i < S) {
      const float al = alpha_w[warp][i];
      float x[8];
      unpack8(source(xs, i, a.n_blocks, pn), x);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = fmaf(al, x[e], acc[e]);
    }
  }
  const uint4 hv = pack8(acc);
  float hf[8];
  unpack8(hv, hf);
  float hss = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) hss = fmaf(hf[e], hf[e], hss);
  if (own) {
    *reinterpret_cast<uint4*>(a.mix + row_off) = hv;
    if (a.commit) {
      *reinterpret_cast<uint4*>(a.blocks + a.n_blocks * blk_stride + row_off) = pn;
      *reinterpret_cast<uint4*>(a.prefix + row_off) = make_uint4(0u, 0u, 0u, 0u);
    } else {
      *reinterpret_cast<uint4*>(a.prefix + row_off) = pn;
    }
  }
  hss = warp_sum(hss);
  if (lane == 0) red2[warp] = hss;
  __syncthreads();
  if (tid < C) {
    float sum = 0.f;
    for (int w = 0; w < nwarps; ++w) sum += red2[w];
    st_async(&part2[c], (uint32_t)tid, sum, &mbar[1]);
  }
  mbar_wait_bounded(&mbar[1]);

  // 6. the RMSNorm of the mixture
  float tot = 0.f;
  for (int k = 0; k < C; ++k) tot += part2[k];
  const float rs = rsqrtf(fmaf(tot, invH, a.eps));
  if (own) {
    float g[8];
    unpack8(gv4, g);
#pragma unroll
    for (int e = 0; e < 8; ++e) hf[e] = hf[e] * rs * g[e];
    *reinterpret_cast<uint4*>(a.y + row_off) = pack8(hf);
  }
}

// Static shared memory of the kernel (the reduction arrays above), kept out of the
// dynamic budget.
constexpr size_t kStaticSmem =
    sizeof(float) * ((kMaxThreads / 32) * 2 * kMaxSources + kMaxCluster * 2 * kMaxSources +
                     (kMaxThreads / 32) * kMaxSources + kMaxThreads / 32 + kMaxCluster);
constexpr size_t kDynSmemLimit = 227 * 1024 - kStaticSmem - 1024;

bool mix_plan(int hidden, int S, MixPlan* p) {
  if (hidden < 8 || hidden > kMaxHidden || hidden % 8) return false;
  if (S < 1 || S > kMaxSources) return false;
  int C = kMaxCluster;
  while (C > 1 && (hidden % (8 * C) != 0 || hidden / C < 128)) C >>= 1;
  const int W = hidden / C;
  const int nv = W / 8;
  int T = (nv + 31) / 32 * 32;
  if (T < 64) T = 64;  // threads 0 .. 2S-1 add the per-source partials
  if (T > kMaxThreads) T = kMaxThreads;
  p->C = C;
  p->W = W;
  if (nv <= kRegThreads) {  // one thread per vector, every operand in registers
    p->reg_smax = S <= 8 ? 8 : S <= 16 ? 16 : 32;
    p->threads = T;
    p->smem = 0;
    return true;
  }
  const size_t smem = (size_t)(S + 4) * W * 2;
  if (smem > kDynSmemLimit) return false;
  p->reg_smax = 0;
  p->threads = T;
  p->smem = smem;
  return true;
}

cudaError_t launch_attnres_mix(const MixArgs& a, const MixPlan& p, cudaStream_t st, bool pdl) {
  // the opt-in above 48 KB counts static and dynamic shared memory together, so it is set
  // once per device whatever this launch's size
  {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    // (setting it twice from racing threads is harmless; the flag only saves the call)
    static std::atomic<int> done[64];
    if (dev < 0 || dev >= 64 || !done[dev].load(std::memory_order_acquire)) {
      e = cudaFuncSetAttribute(k_attnres_mix, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kDynSmemLimit);
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < 64) done[dev].store(1, std::memory_order_release);
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.C, a.R);
  cfg.blockDim = dim3(p.threads);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  int n = 0;
  attr[n].id = cudaLaunchAttributeClusterDimension;
  attr[n].val.clusterDim.x = p.C;
  attr[n].val.clusterDim.y = 1;
  attr[n].val.clusterDim.z = 1;
  ++n;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  switch (p.reg_smax) {
    case 8: return cudaLaunchKernelEx(&cfg, k_attnres_mix_reg<8>, a, p.W, p.C);
    case 16: return cudaLaunchKernelEx(&cfg, k_attnres_mix_reg<16>, a, p.W, p.C);
    case 32: return cudaLaunchKernelEx(&cfg, k_attnres_mix_reg<32>, a, p.W, p.C);
    default: return cudaLaunchKernelEx(&cfg, k_attnres_mix, a, p.W, p.C);
  }
}

cudaError_t mix_status(int* out, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(out, g_mix_status, sizeof(int));
  if (e == cudaSuccess && clear) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_mix_status, &zero, sizeof(int));
  }
  return e;
}

}  // namespace amix
