// k_front.cuh -- device pieces of the front shared by the front kernels (k_front.cu), the
// single persistent launch (k_stream_tc.cu) and the cross-checking forms (k_simple.cu): bf16
// pair arithmetic, add + RMSNorm of a row by one CTA, the warp-per-expert router dot
// products, and top-k + dedup by one CTA.
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

// Power-of-two exponent p such that amax * 2^-p lies in [2^14, 2^15) (0 for amax == 0).
__device__ __forceinline__ int f16_block_exp(float amax) {
  if (!(amax > 0.f)) return 0;
  const int e = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127;
  return max(-100, min(100, e - 14));
}

// 8 bf16 n values (one 16-byte group) -> f16 scaled by `down` (a power of two).
__device__ __forceinline__ uint4 f16_group(uint4 nv, float down) {
  const uint32_t w[4] = {nv.x, nv.y, nv.z, nv.w};
  uint32_t o[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    __half2 h2 = __floats2half2_rn(bf16_lo(w[q]) * down, bf16_hi(w[q]) * down);
    o[q] = *reinterpret_cast<uint32_t*>(&h2);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ float group_amax(uint4 nv) {
  const uint32_t w[4] = {nv.x, nv.y, nv.z, nv.w};
  float m = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[q])), fabsf(bf16_hi(w[q]))));
  return m;
}

// ---------------------------------------------------------------- add + RMSNorm ----
template <int NT>
__device__ __forceinline__ float block_reduce_t(float v, bool is_max, float* part) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = is_max ? warp_max(v) : warp_sum(v);
  __syncthreads();  // part[] may still be read by the previous reduction
  if (lane == 0) part[warp] = v;
  __syncthreads();
  float r = 0.f;
  for (int i = 0; i < NT / 32; ++i) r = is_max ? fmaxf(r, part[i]) : r + part[i];
  return r;
}

// The four E2M1 planes of the 8 n values of group c (16 bytes) of row r, for the
// tensor-core experts: codes to np4 (rows 4r + p), scales as scale-factor atoms to np4a.  A
// 32-element block is the groups of four adjacent lanes (the caller's warps lie wholly inside
// the row's groups or wholly past them), whose maxima are exchanged by shuffles.
__device__ __forceinline__ void store_n_planes(uint4 nv, int r, int c, int H,
                                               uint8_t* __restrict__ np4,
                                               uint8_t* __restrict__ np4a) {
  const uint32_t ww[4] = {nv.x, nv.y, nv.z, nv.w};
  float rv[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    rv[2 * i] = bf16_lo(ww[i]);
    rv[2 * i + 1] = bf16_hi(ww[i]);
  }
#pragma unroll
  for (int pl = 0; pl < 4; ++pl) {
    float am = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) am = fmaxf(am, fabsf(rv[i]));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
    const int e = e2m1_plane_exp(am);
    const float inv = exp2_int(-e), sc = exp2_int(e);
    float xs[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) xs[i] = rv[i] * inv;
    const uint32_t code = e2m1x8_pack(xs);
    uint32_t h[4];
    e2m1x8_to_f16x2(code, h[0], h[1], h[2], h[3]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[i]));
      rv[2 * i] -= f.x * sc;
      rv[2 * i + 1] -= f.y * sc;
    }
    const size_t prow = (size_t)(4 * r + pl);
    reinterpret_cast<uint32_t*>(np4 + prow * (H / 2))[c] = code;
    if ((c & 3) == 0) np4a[sf_atom_offset((int)prow, c / 4)] = (uint8_t)(e + 127);
  }
}

// Add + RMSNorm of row r by a CTA of NT threads (thread i owns the 16-byte groups i, i + NT,
// ... of the row, NG at most, and keeps bf16(x + residual) in registers), gamma already staged
// in shared memory (s_gamma, H / 8 groups).  Two block reductions (sum of squares, then max
// |n| for the f16 copy) in a fixed order; no value is re-read from global memory.  Writes
// r_new and n; the f16 copy of n with its row scale (CUDA-core expert forms, np4 null) or
// the four E2M1 planes of n with their scales in scale-factor atoms (tensor-core forms); the
// shared-expert gate's sigmoid when wsg is given.  part: NT / 32 floats of shared memory.
template <int NT, int NG>
__device__ __forceinline__ void add_rmsnorm_row(
    int r, const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ residual,
    const uint4* s_gamma, __nv_bfloat16* __restrict__ rnew, __nv_bfloat16* __restrict__ n_out,
    __half* __restrict__ n16, float* __restrict__ n16s, int H, float eps,
    const __nv_bfloat16* __restrict__ wsg, float* __restrict__ sgate,
    const float* __restrict__ xpart, int Pk, size_t part_stride, uint8_t* __restrict__ np4,
    uint8_t* __restrict__ np4a, float* part) {
  const int ng = H / 8;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)r * H);
  const uint4* rr = reinterpret_cast<const uint4*>(residual + (size_t)r * H);
  uint4 rn[NG];
  float ss = 0.f;
#pragma unroll
  for (int q = 0; q < NG; ++q) {
    const int c = threadIdx.x + q * NT;
    if (c < ng) {
      uint4 xv;
      if (xpart) {  // x = bf16(the out_proj K parts added in part order)
        const float* p0 = xpart + (size_t)r * H + 8 * (size_t)c;
        float4 a = __ldcg(reinterpret_cast<const float4*>(p0));
        float4 b = __ldcg(reinterpret_cast<const float4*>(p0) + 1);
        for (int pp = 1; pp < Pk; ++pp) {
          const float4* pq = reinterpret_cast<const float4*>(p0 + pp * part_stride);
          const float4 a2 = __ldcg(pq), b2 = __ldcg(pq + 1);
          a.x += a2.x; a.y += a2.y; a.z += a2.z; a.w += a2.w;
          b.x += b2.x; b.y += b2.y; b.z += b2.z; b.w += b2.w;
        }
        xv = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y),
                        pack_bf16x2(b.z, b.w));
      } else {
        xv = xr[c];
      }
      const uint4 rv = rr[c];
      rn[q] = make_uint4(add_bf16x2(xv.x, rv.x), add_bf16x2(xv.y, rv.y), add_bf16x2(xv.z, rv.z),
                         add_bf16x2(xv.w, rv.w));
    } else {
      rn[q] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
#pragma unroll
  for (int q = 0; q < NG; ++q) {
    const uint32_t o[4] = {rn[q].x, rn[q].y, rn[q].z, rn[q].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) ss += bf16_lo(o[i]) * bf16_lo(o[i]) + bf16_hi(o[i]) * bf16_hi(o[i]);
  }
  const float rstd = 1.0f / sqrtf(block_reduce_t<NT>(ss, false, part) / (float)H + eps);
  float down = 1.f;
  if (!np4) {
    // the f16 copy of the CUDA-core expert form, with one power-of-two scale per row (row
    // maximum in [2^14, 2^15)); the tensor-core form takes the E2M1 planes below instead
    float amax = 0.f;
#pragma unroll
    for (int q = 0; q < NG; ++q) {
      const int c = threadIdx.x + q * NT;
      if (c < ng) {
        const uint4 gv = s_gamma[c];
        const uint4 nv = make_uint4(norm_bf16x2(rn[q].x, gv.x, rstd), norm_bf16x2(rn[q].y, gv.y, rstd),
                                    norm_bf16x2(rn[q].z, gv.z, rstd), norm_bf16x2(rn[q].w, gv.w, rstd));
        amax = fmaxf(amax, group_amax(nv));
      }
    }
    const int p = f16_block_exp(block_reduce_t<NT>(amax, true, part));
    down = __uint_as_float((uint32_t)(127 - p) << 23);
    if (threadIdx.x == 0) n16s[r] = __uint_as_float((uint32_t)(127 + p) << 23);
  }
  uint4* rno = reinterpret_cast<uint4*>(rnew + (size_t)r * H);
  uint4* no = reinterpret_cast<uint4*>(n_out + (size_t)r * H);
  uint4* n16o = reinterpret_cast<uint4*>(n16 + (size_t)r * H);
  const uint4* wg4 = reinterpret_cast<const uint4*>(wsg);
  float zg = 0.f;  // this thread's part of the shared-expert gate logit n . wsg
#pragma unroll
  for (int q = 0; q < NG; ++q) {
    const int c = threadIdx.x + q * NT;
    if (c < ng) {
      const uint4 gv = s_gamma[c];
      const uint4 nv = make_uint4(norm_bf16x2(rn[q].x, gv.x, rstd), norm_bf16x2(rn[q].y, gv.y, rstd),
                                  norm_bf16x2(rn[q].z, gv.z, rstd), norm_bf16x2(rn[q].w, gv.w, rstd));
      rno[c] = rn[q];
      no[c] = nv;
      if (!np4) n16o[c] = f16_group(nv, down);
      if (np4) store_n_planes(nv, r, c, H, np4, np4a);
      if (wsg) {
        const uint4 w = __ldg(wg4 + c);
        const uint32_t nn[4] = {nv.x, nv.y, nv.z, nv.w}, ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          zg += bf16_lo(nn[i]) * bf16_lo(ww[i]) + bf16_hi(nn[i]) * bf16_hi(ww[i]);
      }
    }
  }
  if (wsg) {  // the gate of this row: sigmoid of the block-reduced logit
    const float z = block_reduce_t<NT>(zg, false, part);
    if (threadIdx.x == 0) sgate[r] = 1.0f / (1.0f + expf(-z));
  }
}

// Add + RMSNorm of part p of P of row r by a CTA of NT threads (the single persistent launch
// spreads a row over P CTAs): rstd from the whole row (thread-strided 16-byte groups, fixed
// order, then a block reduction; every CTA of the row computes the same), then for the part's
// groups (whole 256-element units, unit range [p U / P, (p + 1) U / P) of U = H / 256)
// r_new, n, the planes of n with their scales, and the part's share of the shared-expert gate
// logit n . wsg into gate_part[p] (when wsg is given).  gamma is read from global memory.
template <int NT>
__device__ __forceinline__ void add_rmsnorm_part(
    int r, int p, int P, const __nv_bfloat16* __restrict__ x,
    const __nv_bfloat16* __restrict__ residual, const __nv_bfloat16* __restrict__ gamma,
    __nv_bfloat16* __restrict__ rnew, __nv_bfloat16* __restrict__ n_out, int H, float eps,
    const __nv_bfloat16* __restrict__ wsg, float* __restrict__ gate_part,
    uint8_t* __restrict__ np4, uint8_t* __restrict__ np4a, float* part) {
  const int ng = H / 8, units = H / 256;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)r * H);
  const uint4* rr = reinterpret_cast<const uint4*>(residual + (size_t)r * H);
  float ss = 0.f;
  for (int c = threadIdx.x; c < ng; c += NT) {
    const uint4 xv = xr[c], rv = rr[c];
    const uint32_t o[4] = {add_bf16x2(xv.x, rv.x), add_bf16x2(xv.y, rv.y),
                           add_bf16x2(xv.z, rv.z), add_bf16x2(xv.w, rv.w)};
#pragma unroll
    for (int i = 0; i < 4; ++i) ss += bf16_lo(o[i]) * bf16_lo(o[i]) + bf16_hi(o[i]) * bf16_hi(o[i]);
  }
  const float rstd = 1.0f / sqrtf(block_reduce_t<NT>(ss, false, part) / (float)H + eps);
  const int c0 = 32 * (p * units / P), c1 = 32 * ((p + 1) * units / P);
  const uint4* g4 = reinterpret_cast<const uint4*>(gamma);
  const uint4* wg4 = reinterpret_cast<const uint4*>(wsg);
  uint4* rno = reinterpret_cast<uint4*>(rnew + (size_t)r * H);
  uint4* no = reinterpret_cast<uint4*>(n_out + (size_t)r * H);
  float zg = 0.f;
  for (int c = c0 + threadIdx.x; c < c1; c += NT) {  // whole warps: c1 - c0 is a multiple of 32
    const uint4 xv = xr[c], rv = rr[c], gv = __ldg(g4 + c);
    const uint4 o = make_uint4(add_bf16x2(xv.x, rv.x), add_bf16x2(xv.y, rv.y),
                               add_bf16x2(xv.z, rv.z), add_bf16x2(xv.w, rv.w));
    const uint4 nv = make_uint4(norm_bf16x2(o.x, gv.x, rstd), norm_bf16x2(o.y, gv.y, rstd),
                                norm_bf16x2(o.z, gv.z, rstd), norm_bf16x2(o.w, gv.w, rstd));
    rno[c] = o;
    no[c] = nv;
    store_n_planes(nv, r, c, H, np4, np4a);
    if (wsg) {
      const uint4 w = __ldg(wg4 + c);
      const uint32_t nn[4] = {nv.x, nv.y, nv.z, nv.w}, ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        zg += bf16_lo(nn[i]) * bf16_lo(ww[i]) + bf16_hi(nn[i]) * bf16_hi(ww[i]);
    }
  }
  if (wsg) {
    const float z = block_reduce_t<NT>(zg, false, part);
    if (threadIdx.x == 0) gate_part[p] = z;
  }
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

// Shared-memory workspace of topk_dedup_block: the picks, each expert's row mask and first
// user slot, and the warps' scan totals (12.5 KB).
struct TopkWs {
  int32_t* s_ids;      // [kMaxPicks]
  uint32_t* rowmask;   // [kMaxExperts]
  int32_t* eoff;       // [kMaxExperts] first user slot of expert e
  int32_t* wsum_d;     // [32]
  int32_t* wsum_u;     // [32]
};
constexpr int kTopkWsBytes = (kMaxPicks + 2 * kMaxExperts + 64) * 4;
// the workspace carved from `base` (4-byte aligned shared memory of kTopkWsBytes)
__device__ __forceinline__ TopkWs topk_ws_at(uint8_t* base) {
  TopkWs w;
  w.s_ids = reinterpret_cast<int32_t*>(base);
  w.rowmask = reinterpret_cast<uint32_t*>(w.s_ids + kMaxPicks);
  w.eoff = reinterpret_cast<int32_t*>(w.rowmask + kMaxExperts);
  w.wsum_d = w.eoff + kMaxExperts;
  w.wsum_u = w.wsum_d + 32;
  return w;
}

template <bool kSmem>
__device__ void topk_dedup_block_ws(const float* logits, int32_t* ids, float* wts,
                                    int32_t* n_distinct, int32_t* uniq, int32_t* user_off,
                                    int32_t* user_list, int32_t* status, int R, int E, int k,
                                    const TopkWs& ws) {
  int32_t* s_ids = ws.s_ids;
  uint32_t* rowmask = ws.rowmask;
  int32_t* eoff = ws.eoff;
  int32_t* wsum_d = ws.wsum_d;
  int32_t* wsum_u = ws.wsum_u;

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

// topk_dedup_block_ws with its workspace in static shared memory.
template <bool kSmem>
__device__ void topk_dedup_block(const float* logits, int32_t* ids, float* wts,
                                 int32_t* n_distinct, int32_t* uniq, int32_t* user_off,
                                 int32_t* user_list, int32_t* status, int R, int E, int k) {
  __shared__ __align__(16) uint8_t ws[kTopkWsBytes];
  topk_dedup_block_ws<kSmem>(logits, ids, wts, n_distinct, uniq, user_off, user_list, status, R,
                             E, k, topk_ws_at(ws));
}

// ------------------------------------------------------------ router on the tensor cores ----
// A router part: 16 experts (M rows of mma.m16n8k16, bf16 x bf16 into fp32) x every row (N,
// four tiles of 8 at most) over K part p of H.  The router kernel runs one part per CTA; the
// single persistent launch runs the parts as virtual CTAs spread over its grid.  The partial
// logits go to scratch; the part whose ticket is the last one adds the parts in part order
// (router_finish), runs top-k and the dedup, and publishes the routing.
constexpr int kRtTile = 16;      // experts per part
constexpr int kRtMaxPart = 2048; // K elements per part at most
constexpr int kRtMaxParts = 16;

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void mma_bf16_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Stage the part's router weights (16 rows of plen bf16, 16-byte row pad) with cp.async,
// one commit group; NTH threads.  They depend on nothing, so this may run before any wait.
template <int NTH>
__device__ __forceinline__ void router_stage_w(uint8_t* sm, const __nv_bfloat16* __restrict__ w_r,
                                               int tile, int p, int plen, int H, int E) {
  const int k0 = p * plen, len = min(plen, H - k0), cpr = len / 8, pitch = plen * 2 + 16;
  const int e0 = tile * kRtTile;
  for (int i = threadIdx.x; i < kRtTile * cpr; i += NTH) {
    const int r = i / cpr, c = i % cpr;
    cp_async16(sm + r * pitch + c * 16, w_r + (size_t)min(e0 + r, E - 1) * H + k0 + c * 8);
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// The rest of part (tile, p) by NW warps: n's rows of the part (cp.async.cg: n may have been
// written earlier in the same launch), the MMAs (warp w takes a slice of the part's
// 32-element K steps; lane (g, t) elements 8t .. 8t+7 of a step for weight rows g, g + 8 and
// activation row g of each N-tile), the warps' tiles added in warp order, the partial logits
// to scratch, then a ticket.  True in the part whose ticket is the last of `total`.
template <int NW>
__device__ __forceinline__ bool router_part(uint8_t* sm, const Scratch& s, int tile, int p,
                                            int plen, int red_off, int R, int H, int E,
                                            uint32_t total, int* s_last) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int k0 = p * plen, len = min(plen, H - k0), cpr = len / 8, pitch = plen * 2 + 16;
  const int e0 = tile * kRtTile;
  uint8_t* sw = sm;                    // [16][pitch] router weights
  uint8_t* sn = sm + kRtTile * pitch;  // [R][pitch] n
  float4* red = reinterpret_cast<float4*>(sm + red_off);  // [NW warps][NT][32 lanes]
  for (int i = tid; i < R * cpr; i += NW * 32) {
    const int r = i / cpr, c = i % cpr;
    cp_async16(sn + r * pitch + c * 16, s.n + (size_t)r * H + k0 + c * 8);
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  const int NT = (R + 7) / 8;  // N-tiles of 8 rows (up to 4)
  const int S = len / 32, spw = (S + NW - 1) / NW;
  float acc[kMaxRows / 8][4];
#pragma unroll
  for (int nt = 0; nt < kMaxRows / 8; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
  const uint8_t* wa = sw + g * pitch + 16 * t;
  const uint8_t* wc = sw + (g + 8) * pitch + 16 * t;
  const uint8_t* nb = sn + 16 * t;
#pragma unroll 1
  for (int st = warp * spw; st < min(S, (warp + 1) * spw); ++st) {
    const uint4 a = *reinterpret_cast<const uint4*>(wa + st * 64);
    const uint4 c = *reinterpret_cast<const uint4*>(wc + st * 64);
#pragma unroll
    for (int nt = 0; nt < kMaxRows / 8; ++nt) {
      if (nt < NT) {
        const uint4 b =
            *reinterpret_cast<const uint4*>(nb + min(8 * nt + g, R - 1) * pitch + st * 64);
        mma_bf16_16816(acc[nt], a.x, c.x, a.y, c.y, b.x, b.y);
        mma_bf16_16816(acc[nt], a.z, c.z, a.w, c.w, b.z, b.w);
      }
    }
  }
  __syncthreads();  // the reduction tiles may overlay the staged tiles every warp has read
#pragma unroll
  for (int nt = 0; nt < kMaxRows / 8; ++nt)
    if (nt < NT)
      red[(warp * NT + nt) * 32 + lane] =
          make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
  __syncthreads();
  if (warp == 0) {
    // lane (g, t): experts g and g + 8, rows 8 nt + 2t and 8 nt + 2t + 1
    for (int nt = 0; nt < NT; ++nt) {
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      for (int w2 = 0; w2 < NW; ++w2) {
        const float4 x = red[(w2 * NT + nt) * 32 + lane];
        v[0] += x.x; v[1] += x.y; v[2] += x.z; v[3] += x.w;
      }
      for (int q = 0; q < 4; ++q) {
        const int e = e0 + g + 8 * (q >> 1), r = 8 * nt + 2 * t + (q & 1);
        if (e < E && r < R) s.logit_parts[((size_t)p * R + r) * E + e] = v[q];
      }
    }
  }
  __threadfence();
  __syncthreads();
  if (tid == 0)
    *s_last = (atomicAdd(&s.counters[kCtrFrontTicket], 1u) == total - 1u) ? 1 : 0;
  __syncthreads();
  return *s_last != 0;
}

// The last part: logits = the P parts added in part order (into shared memory; every part
// of four logits per thread is loaded before any is added), top-k and the dedup, then the
// routing published (every thread's table stores, then the word the expert stages wait for,
// release at GPU scope).  NTH threads; kDynWs: top-k's workspace in `sm` after the logits
// (R E 4 bytes rounded to 16, then kTopkWsBytes), else in static shared memory.
template <int NTH, bool kDynWs>
__device__ __forceinline__ void router_finish(uint8_t* sm, const Scratch& s, int P, int R, int E,
                                              int k) {
  const int tid = threadIdx.x;
  __threadfence();
  float* s_logits = reinterpret_cast<float*>(sm);
  const int RE = R * E;
  constexpr int kJ = 4;
  for (int base = 0; base < RE; base += kJ * NTH) {
    float v[kRtMaxParts][kJ];
#pragma unroll
    for (int pp = 0; pp < kRtMaxParts; ++pp)
#pragma unroll
      for (int j = 0; j < kJ; ++j) {
        const int i = base + tid + j * NTH;
        v[pp][j] = (pp < P && i < RE) ? __ldcg(s.logit_parts + (size_t)pp * RE + i) : 0.f;
      }
#pragma unroll
    for (int j = 0; j < kJ; ++j) {
      float sum = v[0][j];
#pragma unroll
      for (int pp = 1; pp < kRtMaxParts; ++pp)
        if (pp < P) sum += v[pp][j];
      const int i = base + tid + j * NTH;
      if (i < RE) s_logits[i] = sum;
    }
  }
  __syncthreads();
  if (tid == 0) tl_first(s.tl, kTlTopkStart);
  if constexpr (kDynWs)  // the workspace right after the logits in the same shared memory
    topk_dedup_block_ws<true>(s_logits, s.ids, s.wts, s.n_distinct, s.uniq, s.user_off,
                              s.user_list, s.status, R, E, k,
                              topk_ws_at(sm + (((size_t)RE * 4 + 15) & ~(size_t)15)));
  else
    topk_dedup_block<true>(s_logits, s.ids, s.wts, s.n_distinct, s.uniq, s.user_off,
                           s.user_list, s.status, R, E, k);
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    s.counters[kCtrFrontTicket] = 0u;
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(&s.counters[kCtrRouted]), "r"(1u)
                 : "memory");
    tl_first(s.tl, kTlRouted);
  }
}

}  // namespace mtail
