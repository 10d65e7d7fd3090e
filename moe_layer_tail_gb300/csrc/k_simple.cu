// k_simple.cu -- warp-per-output-row CUDA-core kernels for the expert stages and the
// combine.  One warp computes whole dot products for one weight row and every user of it
// (fp32 accumulation in a fixed per-lane order, butterfly reduction), so results do not
// depend on the launch shape.  These kernels are the straightforward form of the stages;
// the streaming kernels in k_stream.cu compute the same values faster.
//
// Sources: "[AMD] integrate kimi k3 monokernel" page, Kernel Replacement table rows "The
// routed experts" (bf16 activations x MXFP4 weights, gate and up, SiLU, down) and "The
// shared expert gate_up / SiLU and mul / down"; "glm53: Long-context indexer ..." page,
// Modifications rows 16 and 20 (each distinct expert once, every using row against it).
#include "k_combine.cuh"
#include "k_front.cuh"
#include "moe_tail_internal.cuh"

namespace mtail {

constexpr int kSimpleWarps = 8;

// 32 MXFP4 elements (16 code bytes) -> 32 floats (unscaled E2M1 values).
__device__ __forceinline__ void dequant32(uint4 c, float* v) {
  uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t h[4];
    e2m1x8_to_f16x2(w[q], h[0], h[1], h[2], h[3]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f = __half22float2(*reinterpret_cast<__half2*>(&h[i]));
      v[q * 8 + i * 2] = f.x;
      v[q * 8 + i * 2 + 1] = f.y;
    }
  }
}

// dot of 32 floats with 32 bf16 activations at p (64 bytes, 16-byte aligned); ordinary loads
// (the CTA's warps share them through L1).
__device__ __forceinline__ float dot32_bf16(const float* v, const __nv_bfloat16* p) {
  const uint4* p4 = reinterpret_cast<const uint4*>(p);
  float a = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 q = p4[c];
    uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      a += v[c * 8 + i * 2] * bf16_lo(w[i]);
      a += v[c * 8 + i * 2 + 1] * bf16_hi(w[i]);
    }
  }
  return a;
}

// Each stage below is a warp-level loop: warp gw of nw (this warp's index among all warps
// of the grid, and their number) takes items gw, gw + nw, ...

// Ask L2 for a weight row's lines before the lanes walk it, so that a warp has the whole row
// in flight rather than one 16-byte block per lane at a time.
__device__ __forceinline__ void prefetch_row(const void* row, size_t bytes, int lane) {
  const char* p = reinterpret_cast<const char*>(row);
  for (size_t o = (size_t)lane * 128; o < bytes; o += 32 * 128)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p + o));
}

// The dots of 32 gate floats and 32 up floats with the same 32 bf16 activations at p, which
// are loaded once for both.
__device__ __forceinline__ void dot32x2_bf16(const float* g, const float* u,
                                             const __nv_bfloat16* p, float& dg, float& du) {
  const uint4* p4 = reinterpret_cast<const uint4*>(p);
  float a = 0.f, b = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 q = p4[c];
    uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      a += g[c * 8 + i * 2] * bf16_lo(w[i]);
      a += g[c * 8 + i * 2 + 1] * bf16_hi(w[i]);
      b += u[c * 8 + i * 2] * bf16_lo(w[i]);
      b += u[c * 8 + i * 2 + 1] * bf16_hi(w[i]);
    }
  }
  dg = a;
  du = b;
}

// Routed gate/up: item (d, j) -> mid[pick, j] for every pick of distinct expert d.
__device__ void routed_gateup_work(long long gw, long long nw, const Dims& dm, const Weights& w,
                                   const Scratch& s) {
  const int lane = threadIdx.x & 31;
  const int D = *s.n_distinct;
  const int H = dm.H, I = dm.I, k = dm.k;
  const long long items = (long long)D * I;
  const int nblk = H / 32;
  for (long long it = gw; it < items; it += nw) {
    const int d = (int)(it / I), j = (int)(it % I);
    const int e = s.uniq[d];
    const int u0 = s.user_off[d], U = s.user_off[d + 1] - u0;
    int rows[kMaxRowsOther];
#pragma unroll
    for (int u = 0; u < kMaxRowsOther; ++u) rows[u] = (u < U) ? s.user_list[u0 + u] / k : 0;
    float ag[kMaxRowsOther], au[kMaxRowsOther];
#pragma unroll
    for (int u = 0; u < kMaxRowsOther; ++u) { ag[u] = 0.f; au[u] = 0.f; }
    const size_t grow = (size_t)e * 2 * I + j, urow = grow + I;
    const uint4* gc = reinterpret_cast<const uint4*>(w.w13c + grow * (H / 2));
    const uint4* uc = reinterpret_cast<const uint4*>(w.w13c + urow * (H / 2));
    const uint8_t* gs = w.w13s + grow * nblk;
    const uint8_t* us = w.w13s + urow * nblk;
    prefetch_row(gc, (size_t)H / 2, lane);
    prefetch_row(uc, (size_t)H / 2, lane);
    prefetch_row(gs, (size_t)nblk, lane);
    prefetch_row(us, (size_t)nblk, lane);
    for (int b = lane; b < nblk; b += 32) {
      float gv[32], uv[32];
      dequant32(__ldg(gc + b), gv);
      dequant32(__ldg(uc + b), uv);
      const float sg = e8m0_to_float(__ldg(gs + b)), su = e8m0_to_float(__ldg(us + b));
#pragma unroll
      for (int u = 0; u < kMaxRowsOther; ++u) {
        if (u < U) {
          float dg, du;
          dot32x2_bf16(gv, uv, s.n + (size_t)rows[u] * H + b * 32, dg, du);
          ag[u] += dg * sg;
          au[u] += du * su;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kMaxRowsOther; ++u) {
      if (u < U) {
        const float g = warp_sum(ag[u]), v = warp_sum(au[u]);
        if (lane == 0) {
          const int pick = s.user_list[u0 + u];
          s.mid[(size_t)pick * I + j] = __float2bfloat16_rn(silu_f(g) * v);
        }
      }
    }
  }
}

// Routed down: item (d, h) -> y[pick, h] for every pick of distinct expert d.
__device__ void routed_down_work(long long gw, long long nw, const Dims& dm, const Weights& w,
                                 const Scratch& s) {
  const int lane = threadIdx.x & 31;
  const int D = *s.n_distinct;
  const int H = dm.H, I = dm.I;
  const long long items = (long long)D * H;
  const int nblk = I / 32;
  for (long long it = gw; it < items; it += nw) {
    const int d = (int)(it / H), h = (int)(it % H);
    const int e = s.uniq[d];
    const int u0 = s.user_off[d], U = s.user_off[d + 1] - u0;
    int picks[kMaxRowsOther];
#pragma unroll
    for (int u = 0; u < kMaxRowsOther; ++u) picks[u] = (u < U) ? s.user_list[u0 + u] : 0;
    float acc[kMaxRowsOther];
#pragma unroll
    for (int u = 0; u < kMaxRowsOther; ++u) acc[u] = 0.f;
    const size_t row = (size_t)e * H + h;
    const uint4* c4 = reinterpret_cast<const uint4*>(w.w2c + row * (I / 2));
    const uint8_t* sc = w.w2s + row * nblk;
    prefetch_row(c4, (size_t)I / 2, lane);
    prefetch_row(sc, (size_t)nblk, lane);
    for (int b = lane; b < nblk; b += 32) {
      float v[32];
      dequant32(__ldg(c4 + b), v);
      const float sb = e8m0_to_float(__ldg(sc + b));
#pragma unroll
      for (int u = 0; u < kMaxRowsOther; ++u)
        if (u < U) acc[u] += dot32_bf16(v, s.mid + (size_t)picks[u] * I + b * 32) * sb;
    }
#pragma unroll
    for (int u = 0; u < kMaxRowsOther; ++u) {
      if (u < U) {
        const float t = warp_sum(acc[u]);
        if (lane == 0) s.y[(size_t)picks[u] * H + h] = t;
      }
    }
  }
}

// Shared gate/up: item j -> ms[r, j] for every row.
__device__ void shared_gateup_work(long long gw, long long nw, const Dims& dm, const Weights& w,
                                   const Scratch& s) {
  const int lane = threadIdx.x & 31;
  const int H = dm.H, Is = dm.Is, R = dm.R;
  for (long long jj = gw; jj < Is; jj += nw) {
    const int j = (int)jj;
    float ag[kMaxRowsOther], au[kMaxRowsOther];
#pragma unroll
    for (int r = 0; r < kMaxRowsOther; ++r) { ag[r] = 0.f; au[r] = 0.f; }
    const uint4* g4 = reinterpret_cast<const uint4*>(w.ws13 + (size_t)j * H);
    const uint4* u4 = reinterpret_cast<const uint4*>(w.ws13 + (size_t)(Is + j) * H);
    prefetch_row(g4, (size_t)H * 2, lane);
    prefetch_row(u4, (size_t)H * 2, lane);
    for (int c = lane; c < H / 8; c += 32) {
      const uint4 gv = __ldg(g4 + c), uv = __ldg(u4 + c);
      const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w}, uw[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
      for (int r = 0; r < kMaxRowsOther; ++r) {
        if (r < R) {
          const uint4 nv = reinterpret_cast<const uint4*>(s.n + (size_t)r * H)[c];
          const uint32_t nw[4] = {nv.x, nv.y, nv.z, nv.w};
          float a = ag[r], b = au[r];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            a += bf16_lo(gw[i]) * bf16_lo(nw[i]); a += bf16_hi(gw[i]) * bf16_hi(nw[i]);
            b += bf16_lo(uw[i]) * bf16_lo(nw[i]); b += bf16_hi(uw[i]) * bf16_hi(nw[i]);
          }
          ag[r] = a; au[r] = b;
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kMaxRowsOther; ++r) {
      if (r < R) {
        const float g = warp_sum(ag[r]), v = warp_sum(au[r]);
        if (lane == 0) s.ms[(size_t)r * Is + j] = __float2bfloat16_rn(silu_f(g) * v);
      }
    }
  }
}

// Shared down: item h -> ys[r, h] for every row.
__device__ void shared_down_work(long long gw, long long nw, const Dims& dm, const Weights& w,
                                 const Scratch& s) {
  const int lane = threadIdx.x & 31;
  const int H = dm.H, Is = dm.Is, R = dm.R;
  for (long long hh = gw; hh < H; hh += nw) {
    const int h = (int)hh;
    float acc[kMaxRowsOther];
#pragma unroll
    for (int r = 0; r < kMaxRowsOther; ++r) acc[r] = 0.f;
    const uint4* w4 = reinterpret_cast<const uint4*>(w.ws2 + (size_t)h * Is);
    prefetch_row(w4, (size_t)Is * 2, lane);
    for (int c = lane; c < Is / 8; c += 32) {
      const uint4 wv = __ldg(w4 + c);
      const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int r = 0; r < kMaxRowsOther; ++r) {
        if (r < R) {
          const uint4 mv = reinterpret_cast<const uint4*>(s.ms + (size_t)r * Is)[c];
          const uint32_t mw[4] = {mv.x, mv.y, mv.z, mv.w};
          float a = acc[r];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            a += bf16_lo(ww[i]) * bf16_lo(mw[i]);
            a += bf16_hi(ww[i]) * bf16_hi(mw[i]);
          }
          acc[r] = a;
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kMaxRowsOther; ++r) {
      if (r < R) {
        const float t = warp_sum(acc[r]);
        if (lane == 0) s.ys[(size_t)r * H + h] = t;
      }
    }
  }
}

#define MT_SIMPLE_KERNEL(name, work)                                                   \
  __global__ void __launch_bounds__(kSimpleWarps * 32) name(Dims dm, Weights w, Scratch s) { \
    work((long long)blockIdx.x * kSimpleWarps + (threadIdx.x >> 5),                      \
         (long long)gridDim.x * kSimpleWarps, dm, w, s);                                 \
  }
MT_SIMPLE_KERNEL(k_shared_gateup_simple, shared_gateup_work)
MT_SIMPLE_KERNEL(k_routed_gateup_simple, routed_gateup_work)
MT_SIMPLE_KERNEL(k_shared_down_simple, shared_down_work)
MT_SIMPLE_KERNEL(k_routed_down_simple, routed_down_work)
#undef MT_SIMPLE_KERNEL

cudaError_t launch_experts_simple(const Dims& d, const Weights& w, const Scratch& s,
                                  int num_sms, cudaStream_t st) {
  const int grid = num_sms * 4;
  k_shared_gateup_simple<<<grid, kSimpleWarps * 32, 0, st>>>(d, w, s);
  k_routed_gateup_simple<<<grid, kSimpleWarps * 32, 0, st>>>(d, w, s);
  k_shared_down_simple<<<grid, kSimpleWarps * 32, 0, st>>>(d, w, s);
  k_routed_down_simple<<<grid, kSimpleWarps * 32, 0, st>>>(d, w, s);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------ combine ----
// out[r, h] = bf16(sum over slots in pick order of wts * y + ys): a fixed-order fp32 sum;
// the residual receives bf16(x + residual), now that every reader of the old value is done.
// One thread per 8 consecutive outputs of a row; the slots' loads are unrolled so that they
// are in flight together.  wait_tiles: instead of waiting for the previous launch as a
// whole, each warp waits (bounded, acquire) until the down items of the two 128-output
// tiles it covers (the shared expert's and one per distinct expert) are counted done.  Before
// that (down_grid > 0, the tensor-core down launch) one thread per CTA waits, polling every
// 2 us, until the down launch's items are all claimed (each of its CTAs then streams its last
// one): the per-tile polls of the whole combine grid, started as soon as the down launch
// begins, had cost the streaming launches up to 18 us a call at 32 rows.

__global__ void __launch_bounds__(256)
k_combine(Dims dm, Scratch s, __nv_bfloat16* __restrict__ out,
          __nv_bfloat16* __restrict__ residual, bool wait_tiles, uint64_t budget_ns,
          bool gated, uint32_t* done, uint32_t seq, const HostArgs* ha, int down_grid) {
  if (!wait_tiles) pdl_wait();
  pdl_trigger();
  if (ha) {  // a host-buffer call: its buffers and number (written before the launch), read
             // once per CTA
    __shared__ const void* s_buf[2];
    __shared__ uint32_t s_seq;
    if (threadIdx.x == 0) {
      s_buf[0] = ha_ptr((const void* const*)&ha->out);
      s_buf[1] = ha_ptr((const void* const*)&ha->residual);
      s_seq = *reinterpret_cast<const volatile uint32_t*>(&ha->seq);
    }
    __syncthreads();
    out = reinterpret_cast<__nv_bfloat16*>(const_cast<void*>(s_buf[0]));
    residual = reinterpret_cast<__nv_bfloat16*>(const_cast<void*>(s_buf[1]));
    seq = s_seq;
  }
  if (threadIdx.x == 0) tl_first(s.tl, kTlCombineStart);
  const int H = dm.H;
  bool claimed = true;
  if (wait_tiles && down_grid > 0) {
    __shared__ int s_claimed;
    if (threadIdx.x == 0) {
      const int D = min(max(__ldcg(s.n_distinct), 1), kMaxPicks);
      const int n_items = (D + 1) * (H / 128);  // the down launch's items
      const uint32_t need = (uint32_t)max(n_items - down_grid, 0);
      s_claimed = wait_count(&s.counters[kCtrDown], need, budget_ns, 2000u) ? 1 : 0;
      if (!s_claimed) set_status(s.status, kStatusTimeout);
    }
    __syncthreads();
    claimed = s_claimed != 0;
  }
  const int ng = H / 8;  // a multiple of 32: whole warps lie in one row
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx < dm.R * ng) {
    const int r = idx / ng, c = idx % ng;
    if (!wait_tiles || (claimed && combine_wait_tiles(s, c, budget_ns)))
      combine_one(dm, s, r, c, out, residual, gated);
    if ((threadIdx.x & 31) == 0) tl_last(s.tl, kTlCombineEnd);
  }
  signal_done(s, done, seq, gridDim.x);
}

cudaError_t launch_combine(const Dims& d, const Scratch& s, __nv_bfloat16* out,
                           __nv_bfloat16* residual, cudaStream_t st, bool pdl, bool wait_tiles,
                           uint64_t budget_ns, bool gated, uint32_t* done, uint32_t seq,
                           const HostArgs* ha, int down_grid) {
  const int n = d.R * d.H / 8;
  return launch_k(k_combine, dim3((n + 255) / 256), dim3(256), 0, st, pdl, d, s, out,
                  residual, wait_tiles, budget_ns, gated, done, seq, ha, down_grid);
}


}  // namespace mtail
