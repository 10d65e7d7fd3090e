// k_front.cuh -- device pieces of the front shared by the front kernels (k_front.cu) and the
// single persistent launch (k_simple.cu): bf16 pair arithmetic, the warp-per-expert router
// dot products, and top-k + dedup by one CTA.
//
// Sources: "[AMD] integrate kimi k3 monokernel" page, Kernel Replacement table rows "The
// post-attention norm", "The router" and "The top-k"; "glm53: Long-context indexer ..."
// page, Modifications table rows 9 (ties run the id reduction only when the maximum is
// shared), 16 and 20 (each distinct expert once, users in row order).
#pragma once

#include "moe_tail.h"
#include "moe_tail_internal.cuh"

namespace mtail {

// Two floats -> two bf16 (round to nearest even) in a word, a in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a)) |
         ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(b)) << 16);
}

// 2 bf16 in a word -> 2 bf16(a + b) in a word (fp32 add, round to nearest even).
__device__ __forceinline__ uint32_t add_bf16x2(uint32_t a, uint32_t b) {
  __nv_bfloat16 lo = __float2bfloat16_rn(bf16_lo(a) + bf16_lo(b));
  __nv_bfloat16 hi = __float2bfloat16_rn(bf16_hi(a) + bf16_hi(b));
  return (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
}
// 2 bf16 r, 2 bf16 gamma -> 2 bf16(r * rstd * gamma)
__device__ __forceinline__ uint32_t norm_bf16x2(uint32_t r, uint32_t g, float rstd) {
  __nv_bfloat16 lo = __float2bfloat16_rn(bf16_lo(r) * rstd * bf16_lo(g));
  __nv_bfloat16 hi = __float2bfloat16_rn(bf16_hi(r) * rstd * bf16_hi(g));
  return (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
}

// Router logits of expert e for every row, by one warp: fp32 accumulation over the lanes'
// strided 8-element chunks of H, butterfly reduction, lane 0 stores logits[r * E + e].  n is
// read with ordinary loads (not the read-only path): the persistent launch writes it
// earlier in the same kernel.
__device__ __forceinline__ void router_warp(const __nv_bfloat16* __restrict__ n,
                                            const __nv_bfloat16* __restrict__ w_r,
                                            float* __restrict__ logits, int R, int H, int E,
                                            int e, int lane) {
  float acc[kMaxRowsOther];
#pragma unroll
  for (int r = 0; r < kMaxRowsOther; ++r) acc[r] = 0.f;
  const uint4* wrow = reinterpret_cast<const uint4*>(w_r + (size_t)e * H);
  const int nch = H / 8;
  for (int c = lane; c < nch; c += 32) {
    uint4 wv = __ldg(wrow + c);
    float wf[8] = {bf16_lo(wv.x), bf16_hi(wv.x), bf16_lo(wv.y), bf16_hi(wv.y),
                   bf16_lo(wv.z), bf16_hi(wv.z), bf16_lo(wv.w), bf16_hi(wv.w)};
#pragma unroll
    for (int r = 0; r < kMaxRowsOther; ++r) {
      if (r < R) {
        uint4 nv = reinterpret_cast<const uint4*>(n + (size_t)r * H)[c];
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
  for (int r = 0; r < kMaxRowsOther; ++r) {
    if (r < R) {
      float v = warp_sum(acc[r]);
      if (lane == 0) logits[(size_t)r * E + e] = v;
    }
  }
}

// ----------------------------------------------------------------- top-k + dedup ----
// Run by one whole CTA.  Warp w ranks rows w, w + nwarps, ...: each round takes the best
// untaken candidate of the row (larger logit, then lower id), so the pick order is (logit
// desc, id asc).  The weights are the softmax of the picked logits.  Then the distinct
// experts of the call are listed in ascending id, with their users in ascending row order
// (an expert appears at most once in a row's picks).

// kSmem: the logits are in this CTA's shared memory (else in global memory, written by an
// earlier launch or by other CTAs of this one before a fence).
template <bool kSmem>
__device__ __forceinline__ float load_logit(const float* l) {
  if constexpr (kSmem) return *l;
  else return __ldcg(l);
}

// Order-preserving 32-bit key of a logit: larger value <=> larger key, +0 and -0 equal; 0
// marks NaN (below every number, -inf included).  key_value inverts it (0 -> NaN).
__device__ __forceinline__ uint32_t order_key(float v) {
  if (v != v) return 0u;
  const uint32_t b = __float_as_uint(v + 0.0f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

// The k largest logits of one row, for one warp: lane i < k returns pick i (value, id), in
// descending order, ties to the lower id.  The row's keys sit lane-strided in registers (Q
// slots per lane, Q * 32 >= E); each lane keeps its best untaken candidate, a pick is one
// warp max over the lanes' best keys and one warp min over the ids holding it, and only the
// lane that owned the pick looks at its slots again.  If only NaN candidates are left the
// lowest untaken id is taken and the status flags the routing.
template <bool kSmem, int Q>
__device__ __forceinline__ void topk_row(const float* l, int E, int k, int32_t* status,
                                         float& pv, int& pe) {
  const int lane = threadIdx.x & 31;
  uint32_t key[Q];
  uint32_t tk = 0u;  // bit q: slot q taken (or past E)
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    const int e = lane + 32 * q;
    key[q] = (e < E) ? order_key(load_logit<kSmem>(l + e)) : 0u;
    if (e >= E) tk |= 1u << q;
  }
  uint32_t bk = 0u;  // this lane's best untaken candidate (key, id)
  uint32_t be = 0xffffffffu;
#pragma unroll
  for (int q = 0; q < Q; ++q)
    if (!((tk >> q) & 1u) && (key[q] > bk || be == 0xffffffffu)) { bk = key[q]; be = lane + 32 * q; }
  pv = 0.f;
  pe = 0;
  for (int i = 0; i < k; ++i) {
    const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
    const uint32_t we = __reduce_min_sync(0xffffffffu, bk == mk ? be : 0xffffffffu);
    if (mk == 0u && lane == 0) set_status(status, kStatusBadRouting);
    if ((int)(we & 31u) == lane) {
      tk |= 1u << (we >> 5);
      bk = 0u;
      be = 0xffffffffu;
#pragma unroll
      for (int q = 0; q < Q; ++q)
        if (!((tk >> q) & 1u) && (key[q] > bk || be == 0xffffffffu)) { bk = key[q]; be = lane + 32 * q; }
    }
    if (lane == i) { pv = key_value(mk); pe = (int)we; }
  }
}

// Compare-exchange of two (key, id) candidates so that the better one (larger key, then
// lower id) comes first.
__device__ __forceinline__ void cas_desc(uint32_t& ka, uint32_t& ia, uint32_t& kb, uint32_t& ib) {
  const bool sw = kb > ka || (kb == ka && ib < ia);
  const uint32_t k0 = sw ? kb : ka, i0 = sw ? ib : ia;
  kb = sw ? ka : kb;
  ib = sw ? ia : ib;
  ka = k0;
  ia = i0;
}

// topk_row for E <= 256: each lane first sorts its 8 candidates (best first) with Batcher's
// 19-comparator network, so that handing over a pick costs its owner a shift of the list
// instead of a rescan.  Slots past E are (key 0, id ~0): after every expert, NaN ones
// included, and never picked.
template <bool kSmem>
__device__ __forceinline__ void topk_row_sorted(const float* l, int E, int k, int32_t* status,
                                                float& pv, int& pe) {
  const int lane = threadIdx.x & 31;
  uint32_t key[8], id[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int e = lane + 32 * q;
    key[q] = (e < E) ? order_key(load_logit<kSmem>(l + e)) : 0u;
    id[q] = (e < E) ? (uint32_t)e : 0xffffffffu;
  }
#define MT_CAS(a, b) cas_desc(key[a], id[a], key[b], id[b])
  MT_CAS(0, 1); MT_CAS(2, 3); MT_CAS(4, 5); MT_CAS(6, 7);
  MT_CAS(0, 2); MT_CAS(1, 3); MT_CAS(4, 6); MT_CAS(5, 7);
  MT_CAS(1, 2); MT_CAS(5, 6);
  MT_CAS(0, 4); MT_CAS(1, 5); MT_CAS(2, 6); MT_CAS(3, 7);
  MT_CAS(2, 4); MT_CAS(3, 5);
  MT_CAS(1, 2); MT_CAS(3, 4); MT_CAS(5, 6);
#undef MT_CAS
  pv = 0.f;
  pe = 0;
  for (int i = 0; i < k; ++i) {
    const uint32_t mk = __reduce_max_sync(0xffffffffu, key[0]);
    const uint32_t we = __reduce_min_sync(0xffffffffu, key[0] == mk ? id[0] : 0xffffffffu);
    if (mk == 0u && lane == 0) set_status(status, kStatusBadRouting);
    if (id[0] == we) {  // this lane owned the pick: the next candidate moves up
#pragma unroll
      for (int q = 0; q < 7; ++q) {
        key[q] = key[q + 1];
        id[q] = id[q + 1];
      }
      key[7] = 0u;
      id[7] = 0xffffffffu;
    }
    if (lane == i) { pv = key_value(mk); pe = (int)we; }
  }
}

template <bool kSmem>
__device__ void topk_dedup_block(const float* logits, int32_t* ids, float* wts,
                                 int32_t* n_distinct, int32_t* uniq, int32_t* user_off,
                                 int32_t* user_list, int32_t* status, int R, int E, int k) {
  __shared__ int32_t s_ids[kMaxPicks];
  __shared__ uint32_t rowmask[kMaxExperts];
  __shared__ int32_t eoff[kMaxExperts];  // first user slot of expert e
  __shared__ int32_t wsum_d[32], wsum_u[32];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthreads = blockDim.x, nwarps = nthreads >> 5;
  for (int e = tid; e < E; e += nthreads) rowmask[e] = 0u;

  for (int row = warp; row < R; row += nwarps) {
    const float* l = logits + (size_t)row * E;
    float pv;  // lane i < k keeps pick i
    int pe;
    if (E <= 256) topk_row_sorted<kSmem>(l, E, k, status, pv, pe);
    else if (E <= 512) topk_row<kSmem, 16>(l, E, k, status, pv, pe);
    else topk_row<kSmem, kMaxExperts / 32>(l, E, k, status, pv, pe);
    // weights: softmax of the picked logits (lane i holds pick i; pick 0 is the largest)
    const float m = __shfl_sync(0xffffffffu, pv, 0);
    const float ex = (lane < k) ? expf(pv - m) : 0.f;
    const float z = warp_sum(ex);
    if (lane < k) {
      wts[row * k + lane] = ex / z;
      ids[row * k + lane] = pe;
      s_ids[row * k + lane] = pe;
    }
  }
  __syncthreads();
  for (int p = tid; p < R * k; p += nthreads) atomicOr(&rowmask[s_ids[p]], 1u << (p / k));
  __syncthreads();
  // exclusive scans over experts of (used ? 1 : 0) and popc(rowmask): each thread owns
  // `per` consecutive experts; warp scan, then warp totals in warp order
  const int per = (E + nthreads - 1) / nthreads;
  const int e0 = tid * per;
  int cd = 0, cu = 0;
  for (int q = 0; q < per; ++q) {
    const int e = e0 + q;
    if (e < E && rowmask[e]) { cd += 1; cu += __popc(rowmask[e]); }
  }
  int id_ = cd, iu = cu;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int td = __shfl_up_sync(0xffffffffu, id_, o);
    const int tu = __shfl_up_sync(0xffffffffu, iu, o);
    if (lane >= o) { id_ += td; iu += tu; }
  }
  if (lane == 31) { wsum_d[warp] = id_; wsum_u[warp] = iu; }
  __syncthreads();
  int bd = 0, bu = 0;
  for (int w2 = 0; w2 < warp; ++w2) { bd += wsum_d[w2]; bu += wsum_u[w2]; }
  int xd = bd + id_ - cd, xu = bu + iu - cu;  // exclusive prefixes at e0
  for (int q = 0; q < per; ++q) {
    const int e = e0 + q;
    if (e < E && rowmask[e]) {
      eoff[e] = xu;
      uniq[xd] = e;
      user_off[xd] = xu;
      xd += 1;
      xu += __popc(rowmask[e]);
    }
  }
  if (tid == nthreads - 1) {
    const int D = bd + id_, U = bu + iu;
    if (D < 1 || D > R * k || U != R * k) set_status(status, kStatusBadDistinct);
    *n_distinct = D;
    user_off[D] = U;
  }
  __syncthreads();
  // place each pick at its expert's slot: users of an expert are in ascending row order
  for (int p = tid; p < R * k; p += nthreads) {
    const int e = s_ids[p], r = p / k;
    const int rank = __popc(rowmask[e] & ((1u << r) - 1u));
    user_list[eoff[e] + rank] = p;
  }
}

}  // namespace mtail
