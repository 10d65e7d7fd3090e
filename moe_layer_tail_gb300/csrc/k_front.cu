// k_front.cu -- the front of the tail: residual add + RMSNorm, router GEMV, top-k and the
// expert dedup that builds the call's work list.
//
// Sources: "[AMD] integrate kimi k3 monokernel" page, Kernel Replacement table rows "The
// post-attention norm", "The router" and "The top-k"; "glm53: Long-context indexer ..."
// page, Modifications table rows 9 (ties run the id reduction only when the maximum is
// shared), 10 (bf16 activations before the router), 16 and 20 (each distinct expert once,
// users in row order).
#include "moe_tail_internal.cuh"

namespace mtail {

// ---------------------------------------------------------------- add + RMSNorm ----
// One CTA per row.  Each thread owns whole 32-element blocks, so the per-block f16 scale
// of the routed experts' activation copy is thread-local.  The residual is rewritten in
// place by the thread that read it.
constexpr int kNormThreads = 256;

__global__ void __launch_bounds__(kNormThreads)
k_add_rmsnorm(const __nv_bfloat16* __restrict__ x, __nv_bfloat16* __restrict__ residual,
              const __nv_bfloat16* __restrict__ gamma, __nv_bfloat16* __restrict__ n_out,
              __half* __restrict__ n16, float* __restrict__ n16s, uint32_t* __restrict__ counters,
              int H, float eps) {
  const int r = blockIdx.x;
  if (r == 0 && threadIdx.x < 8) counters[threadIdx.x] = 0u;  // work counters of this call
  const int nblk = H / 32;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)r * H);
  uint4* rr = reinterpret_cast<uint4*>(residual + (size_t)r * H);
  float ss = 0.f;
  for (int b = threadIdx.x; b < nblk; b += kNormThreads) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint4 xv = xr[b * 4 + c], rv = rr[b * 4 + c];
      uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, rw[4] = {rv.x, rv.y, rv.z, rv.w}, ow[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        __nv_bfloat16 lo = __float2bfloat16_rn(bf16_lo(xw[q]) + bf16_lo(rw[q]));
        __nv_bfloat16 hi = __float2bfloat16_rn(bf16_hi(xw[q]) + bf16_hi(rw[q]));
        float flo = __bfloat162float(lo), fhi = __bfloat162float(hi);
        ss += flo * flo + fhi * fhi;
        ow[q] = (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
      }
      rr[b * 4 + c] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
    }
  }
  // deterministic block reduction: butterfly in each warp, then warp partials in order
  __shared__ float part[kNormThreads / 32];
  __shared__ float s_rstd;
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int i = 0; i < kNormThreads / 32; ++i) t += part[i];
    s_rstd = 1.0f / sqrtf(t / (float)H + eps);
  }
  __syncthreads();
  const float rstd = s_rstd;
  const uint4* g4 = reinterpret_cast<const uint4*>(gamma);
  uint4* no = reinterpret_cast<uint4*>(n_out + (size_t)r * H);
  uint4* n16o = reinterpret_cast<uint4*>(n16 + (size_t)r * H);
  for (int b = threadIdx.x; b < nblk; b += kNormThreads) {
    float v[32];
    float amax = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint4 rv = rr[b * 4 + c], gv = g4[b * 4 + c];
      uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w}, ow[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        __nv_bfloat16 lo = __float2bfloat16_rn(bf16_lo(rw[q]) * rstd * bf16_lo(gw[q]));
        __nv_bfloat16 hi = __float2bfloat16_rn(bf16_hi(rw[q]) * rstd * bf16_hi(gw[q]));
        v[c * 8 + q * 2] = __bfloat162float(lo);
        v[c * 8 + q * 2 + 1] = __bfloat162float(hi);
        amax = fmaxf(amax, fmaxf(fabsf(v[c * 8 + q * 2]), fabsf(v[c * 8 + q * 2 + 1])));
        ow[q] = (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
      }
      no[b * 4 + c] = make_uint4(ow[0], ow[1], ow[2], ow[3]);
    }
    // f16 copy scaled by 2^-p so that the block maximum lies in [2^14, 2^15): exact for
    // every bf16 value down to 2^-29 of the block maximum.
    int p = 0;
    if (amax > 0.f) {
      int e = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127;
      p = max(-100, min(100, e - 14));
    }
    const float down = __uint_as_float((uint32_t)(127 - p) << 23);
    n16s[(size_t)r * nblk + b] = __uint_as_float((uint32_t)(127 + p) << 23);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t hw[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        __half2 h2 = __floats2half2_rn(v[c * 8 + q * 2] * down, v[c * 8 + q * 2 + 1] * down);
        hw[q] = *reinterpret_cast<uint32_t*>(&h2);
      }
      n16o[b * 4 + c] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    }
  }
}

cudaError_t launch_add_rmsnorm(const Dims& d, const __nv_bfloat16* x, __nv_bfloat16* residual,
                               const Weights& w, const Scratch& s, cudaStream_t st) {
  k_add_rmsnorm<<<d.R, kNormThreads, 0, st>>>(x, residual, w.gamma, s.n, s.n16, s.n16s,
                                              s.counters, d.H, d.eps);
  return cudaGetLastError();
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
  if (e >= E) return;
  float acc[kMaxRows];
#pragma unroll
  for (int r = 0; r < kMaxRows; ++r) acc[r] = 0.f;
  const uint4* wrow = reinterpret_cast<const uint4*>(w_r + (size_t)e * H);
  const int nch = H / 8;
  for (int c = lane; c < nch; c += 32) {
    uint4 wv = __ldg(wrow + c);
    float wf[8] = {bf16_lo(wv.x), bf16_hi(wv.x), bf16_lo(wv.y), bf16_hi(wv.y),
                   bf16_lo(wv.z), bf16_hi(wv.z), bf16_lo(wv.w), bf16_hi(wv.w)};
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) {
      if (r < R) {
        uint4 nv = __ldg(reinterpret_cast<const uint4*>(n + (size_t)r * H) + c);
        float a = acc[r];
        a += wf[0] * bf16_lo(nv.x); a += wf[1] * bf16_hi(nv.x);
        a += wf[2] * bf16_lo(nv.y); a += wf[3] * bf16_hi(nv.y);
        a += wf[4] * bf16_lo(nv.z); a += wf[5] * bf16_hi(nv.z);
        a += wf[6] * bf16_lo(nv.w); a += wf[7] * bf16_hi(nv.w);
        acc[r] = a;
      }
    }
  }
#pragma unroll
  for (int r = 0; r < kMaxRows; ++r) {
    if (r < R) {
      float v = warp_sum(acc[r]);
      if (lane == 0) logits[(size_t)r * E + e] = v;
    }
  }
}

cudaError_t launch_router(const Dims& d, const Weights& w, const Scratch& s, cudaStream_t st) {
  dim3 grid((d.E + kRouterWarps - 1) / kRouterWarps);
  k_router<<<grid, kRouterWarps * 32, 0, st>>>(s.n, w.w_r, s.logits, d.R, d.H, d.E);
  return cudaGetLastError();
}

// ----------------------------------------------------------------- top-k + dedup ----
// One CTA.  Warp r ranks row r: each round every lane takes its best untaken candidate
// (larger logit, then lower id) and a butterfly over (value, id) pairs finds the round's
// pick; an exact tie of the value resolves to the lower id, so the pick order is the
// order of (logit desc, id asc).  The weights are the softmax of the picked logits.
// Then the distinct experts of the call are listed in ascending id, with their users in
// ascending row order (an expert appears at most once in a row's picks).
constexpr int kTopkThreads = 512;

__device__ __forceinline__ bool better(float v, int e, float bv, int be) {
  return v > bv || (v == bv && e < be);
}

__global__ void __launch_bounds__(kTopkThreads)
k_topk_dedup(const float* __restrict__ logits, int32_t* __restrict__ ids,
             float* __restrict__ wts, int32_t* __restrict__ n_distinct,
             int32_t* __restrict__ uniq, int32_t* __restrict__ user_off,
             int32_t* __restrict__ user_list, int32_t* __restrict__ status, int R, int E,
             int k) {
  __shared__ uint32_t taken[kMaxRows][kMaxExperts / 32];
  __shared__ float pickv[kMaxRows][kMaxTopK];
  __shared__ int32_t s_ids[kMaxPicks];
  __shared__ uint32_t rowmask[kMaxExperts];
  __shared__ int32_t eoff[kMaxExperts];   // first user slot of expert e
  __shared__ int32_t wsum_d[kTopkThreads / 32], wsum_u[kTopkThreads / 32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < kMaxRows * (kMaxExperts / 32); i += kTopkThreads)
    (&taken[0][0])[i] = 0u;
  for (int e = tid; e < kMaxExperts; e += kTopkThreads) rowmask[e] = 0u;
  __syncthreads();

  if (warp < R) {
    const float* l = logits + (size_t)warp * E;
    for (int i = 0; i < k; ++i) {
      float bv = -INFINITY;
      int be = 0x7fffffff;
      for (int e = lane; e < E; e += 32) {
        if (taken[warp][e >> 5] & (1u << (e & 31))) continue;
        float v = l[e];
        if (better(v, e, bv, be)) { bv = v; be = e; }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        int oe = __shfl_xor_sync(0xffffffffu, be, o);
        if (better(ov, oe, bv, be)) { bv = ov; be = oe; }
      }
      if (be >= E) {  // only NaN candidates left: take the lowest untaken id, flag it
        be = E - 1;  // unreachable fallback: some id is always untaken while i < k <= E
        for (int e = 0; e < E; ++e)
          if (!(taken[warp][e >> 5] & (1u << (e & 31)))) { be = e; break; }
        bv = -INFINITY;
        if (lane == 0) set_status(status, kStatusBadRouting);
      }
      if (lane == 0) {
        taken[warp][be >> 5] |= 1u << (be & 31);
        pickv[warp][i] = l[be];
        s_ids[warp * k + i] = be;
      }
      __syncwarp();
    }
    if (lane == 0) {
      float m = pickv[warp][0], z = 0.f;
      for (int i = 0; i < k; ++i) z += expf(pickv[warp][i] - m);
      for (int i = 0; i < k; ++i) {
        wts[warp * k + i] = expf(pickv[warp][i] - m) / z;
        ids[warp * k + i] = s_ids[warp * k + i];
      }
    }
  }
  __syncthreads();
  // rows using each expert
  for (int p = tid; p < R * k; p += kTopkThreads)
    atomicOr(&rowmask[s_ids[p]], 1u << (p / k));
  __syncthreads();
  // exclusive scans over experts of (used ? 1 : 0) and popc(rowmask): block of 512
  // threads, two experts per thread, scan of warp totals in warp order.
  const int e0 = tid * 2;
  int cd = 0, cu = 0;
  for (int q = 0; q < 2; ++q) {
    int e = e0 + q;
    if (e < E && rowmask[e]) { cd += 1; cu += __popc(rowmask[e]); }
  }
  int id_ = cd, iu = cu;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int td = __shfl_up_sync(0xffffffffu, id_, o), tu = __shfl_up_sync(0xffffffffu, iu, o);
    if (lane >= o) { id_ += td; iu += tu; }
  }
  if (lane == 31) { wsum_d[warp] = id_; wsum_u[warp] = iu; }
  __syncthreads();
  int bd = 0, bu = 0;
  for (int w2 = 0; w2 < warp; ++w2) { bd += wsum_d[w2]; bu += wsum_u[w2]; }
  int xd = bd + id_ - cd, xu = bu + iu - cu;  // exclusive prefixes at e0
  for (int q = 0; q < 2; ++q) {
    int e = e0 + q;
    if (e < E && rowmask[e]) {
      eoff[e] = xu;
      uniq[xd] = e;
      user_off[xd] = xu;
      xd += 1;
      xu += __popc(rowmask[e]);
    }
  }
  if (tid == kTopkThreads - 1) {
    int D = bd + id_, U = bu + iu;
    if (D < 1 || D > R * k || U != R * k) set_status(status, kStatusBadDistinct);
    *n_distinct = D;
    user_off[D] = U;
  }
  __syncthreads();
  // place each pick at its expert's slot: users of an expert are in ascending row order
  for (int p = tid; p < R * k; p += kTopkThreads) {
    int e = s_ids[p], r = p / k;
    int rank = __popc(rowmask[e] & ((1u << r) - 1u));
    user_list[eoff[e] + rank] = p;
  }
}

cudaError_t launch_topk_dedup(const Dims& d, const Scratch& s, cudaStream_t st) {
  k_topk_dedup<<<1, kTopkThreads, 0, st>>>(s.logits, s.ids, s.wts, s.n_distinct, s.uniq,
                                           s.user_off, s.user_list, s.status, d.R, d.E, d.k);
  return cudaGetLastError();
}

}  // namespace mtail
