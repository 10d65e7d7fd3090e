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

// dot of 32 floats with 32 bf16 values at p (64 bytes, 16-byte aligned)
__device__ __forceinline__ float dot32_bf16(const float* v, const __nv_bfloat16* p) {
  const uint4* p4 = reinterpret_cast<const uint4*>(p);
  float a = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 q = __ldg(p4 + c);
    uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      a += v[c * 8 + i * 2] * bf16_lo(w[i]);
      a += v[c * 8 + i * 2 + 1] * bf16_hi(w[i]);
    }
  }
  return a;
}

// Routed gate/up: item (d, j) -> mid[pick, j] for every pick of distinct expert d.
__global__ void __launch_bounds__(kSimpleWarps * 32)
k_routed_gateup_simple(Dims dm, Weights w, Scratch s) {
  const int lane = threadIdx.x & 31;
  const int D = *s.n_distinct;
  const int H = dm.H, I = dm.I, k = dm.k;
  const long long items = (long long)D * I;
  const int nblk = H / 32;
  for (long long it = (long long)blockIdx.x * kSimpleWarps + (threadIdx.x >> 5); it < items;
       it += (long long)gridDim.x * kSimpleWarps) {
    const int d = (int)(it / I), j = (int)(it % I);
    const int e = s.uniq[d];
    const int u0 = s.user_off[d], U = s.user_off[d + 1] - u0;
    int rows[kMaxRows];
#pragma unroll
    for (int u = 0; u < kMaxRows; ++u) rows[u] = (u < U) ? s.user_list[u0 + u] / k : 0;
    float ag[kMaxRows], au[kMaxRows];
#pragma unroll
    for (int u = 0; u < kMaxRows; ++u) { ag[u] = 0.f; au[u] = 0.f; }
    const size_t grow = (size_t)e * 2 * I + j, urow = grow + I;
    const uint4* gc = reinterpret_cast<const uint4*>(w.w13c + grow * (H / 2));
    const uint4* uc = reinterpret_cast<const uint4*>(w.w13c + urow * (H / 2));
    const uint8_t* gs = w.w13s + grow * nblk;
    const uint8_t* us = w.w13s + urow * nblk;
    for (int b = lane; b < nblk; b += 32) {
      float gv[32], uv[32];
      dequant32(__ldg(gc + b), gv);
      dequant32(__ldg(uc + b), uv);
      const float sg = e8m0_to_float(__ldg(gs + b)), su = e8m0_to_float(__ldg(us + b));
#pragma unroll
      for (int u = 0; u < kMaxRows; ++u) {
        if (u < U) {
          const __nv_bfloat16* np = s.n + (size_t)rows[u] * H + b * 32;
          ag[u] += dot32_bf16(gv, np) * sg;
          au[u] += dot32_bf16(uv, np) * su;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kMaxRows; ++u) {
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
__global__ void __launch_bounds__(kSimpleWarps * 32)
k_routed_down_simple(Dims dm, Weights w, Scratch s) {
  const int lane = threadIdx.x & 31;
  const int D = *s.n_distinct;
  const int H = dm.H, I = dm.I;
  const long long items = (long long)D * H;
  const int nblk = I / 32;
  for (long long it = (long long)blockIdx.x * kSimpleWarps + (threadIdx.x >> 5); it < items;
       it += (long long)gridDim.x * kSimpleWarps) {
    const int d = (int)(it / H), h = (int)(it % H);
    const int e = s.uniq[d];
    const int u0 = s.user_off[d], U = s.user_off[d + 1] - u0;
    int picks[kMaxRows];
#pragma unroll
    for (int u = 0; u < kMaxRows; ++u) picks[u] = (u < U) ? s.user_list[u0 + u] : 0;
    float acc[kMaxRows];
#pragma unroll
    for (int u = 0; u < kMaxRows; ++u) acc[u] = 0.f;
    const size_t row = (size_t)e * H + h;
    const uint4* c4 = reinterpret_cast<const uint4*>(w.w2c + row * (I / 2));
    const uint8_t* sc = w.w2s + row * nblk;
    for (int b = lane; b < nblk; b += 32) {
      float v[32];
      dequant32(__ldg(c4 + b), v);
      const float sb = e8m0_to_float(__ldg(sc + b));
#pragma unroll
      for (int u = 0; u < kMaxRows; ++u)
        if (u < U) acc[u] += dot32_bf16(v, s.mid + (size_t)picks[u] * I + b * 32) * sb;
    }
#pragma unroll
    for (int u = 0; u < kMaxRows; ++u) {
      if (u < U) {
        const float t = warp_sum(acc[u]);
        if (lane == 0) s.y[(size_t)picks[u] * H + h] = t;
      }
    }
  }
}

// Shared gate/up: item j -> ms[r, j] for every row.
__global__ void __launch_bounds__(kSimpleWarps * 32)
k_shared_gateup_simple(Dims dm, Weights w, Scratch s) {
  const int lane = threadIdx.x & 31;
  const int H = dm.H, Is = dm.Is, R = dm.R;
  for (int j = blockIdx.x * kSimpleWarps + (threadIdx.x >> 5); j < Is;
       j += gridDim.x * kSimpleWarps) {
    float ag[kMaxRows], au[kMaxRows];
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) { ag[r] = 0.f; au[r] = 0.f; }
    const uint4* g4 = reinterpret_cast<const uint4*>(w.ws13 + (size_t)j * H);
    const uint4* u4 = reinterpret_cast<const uint4*>(w.ws13 + (size_t)(Is + j) * H);
    for (int c = lane; c < H / 8; c += 32) {
      const uint4 gv = __ldg(g4 + c), uv = __ldg(u4 + c);
      const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w}, uw[4] = {uv.x, uv.y, uv.z, uv.w};
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r) {
        if (r < R) {
          const uint4 nv = __ldg(reinterpret_cast<const uint4*>(s.n + (size_t)r * H) + c);
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
    for (int r = 0; r < kMaxRows; ++r) {
      if (r < R) {
        const float g = warp_sum(ag[r]), v = warp_sum(au[r]);
        if (lane == 0) s.ms[(size_t)r * Is + j] = __float2bfloat16_rn(silu_f(g) * v);
      }
    }
  }
}

// Shared down: item h -> ys[r, h] for every row.
__global__ void __launch_bounds__(kSimpleWarps * 32)
k_shared_down_simple(Dims dm, Weights w, Scratch s) {
  const int lane = threadIdx.x & 31;
  const int H = dm.H, Is = dm.Is, R = dm.R;
  for (int h = blockIdx.x * kSimpleWarps + (threadIdx.x >> 5); h < H;
       h += gridDim.x * kSimpleWarps) {
    float acc[kMaxRows];
#pragma unroll
    for (int r = 0; r < kMaxRows; ++r) acc[r] = 0.f;
    const uint4* w4 = reinterpret_cast<const uint4*>(w.ws2 + (size_t)h * Is);
    for (int c = lane; c < Is / 8; c += 32) {
      const uint4 wv = __ldg(w4 + c);
      const uint32_t ww[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
      for (int r = 0; r < kMaxRows; ++r) {
        if (r < R) {
          const uint4 mv = __ldg(reinterpret_cast<const uint4*>(s.ms + (size_t)r * Is) + c);
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
    for (int r = 0; r < kMaxRows; ++r) {
      if (r < R) {
        const float t = warp_sum(acc[r]);
        if (lane == 0) s.ys[(size_t)r * H + h] = t;
      }
    }
  }
}

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
// tiles it covers (the shared expert's and one per distinct expert) are counted done.
__global__ void __launch_bounds__(256)
k_combine(Dims dm, Scratch s, __nv_bfloat16* __restrict__ out,
          __nv_bfloat16* __restrict__ residual, bool wait_tiles, uint64_t budget_ns,
          bool gated) {
  if (!wait_tiles) pdl_wait();
  pdl_trigger();
  const int H = dm.H, k = dm.k;
  const int ng = H / 8;  // a multiple of 32: whole warps lie in one row
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= dm.R * ng) return;
  const int r = idx / ng, c = idx % ng;
  if (wait_tiles) {
    const int lane = threadIdx.x & 31;
    const uint32_t need = (uint32_t)min(max(*s.n_distinct, 1), kMaxPicks) + 1u;
    bool ok = true;
    if ((lane & 15) == 0) ok = wait_count(&s.counters[kCtrTileDone + c / 16], need, budget_ns);
    if (__any_sync(0xffffffffu, !ok)) {
      if (lane == 0) set_status(s.status, kStatusTimeout);
      return;
    }
    __syncwarp();  // orders the other lanes' loads after lanes 0 and 16's acquires
  }
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int i0 = 0; i0 < k; i0 += 8) {
    float4 ya[8], yb[8];
    float wv[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int i = i0 + j;
      if (i < k) {
        const float4* yp = reinterpret_cast<const float4*>(s.y + (size_t)(r * k + i) * H) + 2 * c;
        ya[j] = __ldcg(yp);
        yb[j] = __ldcg(yp + 1);
        wv[j] = s.wts[r * k + i];
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (i0 + j < k) {
        acc[0] += wv[j] * ya[j].x; acc[1] += wv[j] * ya[j].y;
        acc[2] += wv[j] * ya[j].z; acc[3] += wv[j] * ya[j].w;
        acc[4] += wv[j] * yb[j].x; acc[5] += wv[j] * yb[j].y;
        acc[6] += wv[j] * yb[j].z; acc[7] += wv[j] * yb[j].w;
      }
    }
  }
  // + the shared expert's output, times its row's sigmoid gate when the layer has one
  const float4* ysp = reinterpret_cast<const float4*>(s.ys + (size_t)r * H) + 2 * c;
  const float4 s0 = __ldcg(ysp), s1 = __ldcg(ysp + 1);
  const float gt = gated ? __ldcg(s.sgate + r) : 1.f;
  acc[0] = fmaf(gt, s0.x, acc[0]); acc[1] = fmaf(gt, s0.y, acc[1]);
  acc[2] = fmaf(gt, s0.z, acc[2]); acc[3] = fmaf(gt, s0.w, acc[3]);
  acc[4] = fmaf(gt, s1.x, acc[4]); acc[5] = fmaf(gt, s1.y, acc[5]);
  acc[6] = fmaf(gt, s1.z, acc[6]); acc[7] = fmaf(gt, s1.w, acc[7]);
  uint32_t o[4];
#pragma unroll
  for (int q = 0; q < 4; ++q)
    o[q] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * q])) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc[2 * q + 1])) << 16);
  reinterpret_cast<uint4*>(out + (size_t)r * H)[c] = make_uint4(o[0], o[1], o[2], o[3]);
  reinterpret_cast<uint4*>(residual + (size_t)r * H)[c] =
      __ldcg(reinterpret_cast<const uint4*>(s.rnew + (size_t)r * H) + c);
}

cudaError_t launch_combine(const Dims& d, const Scratch& s, __nv_bfloat16* out,
                           __nv_bfloat16* residual, cudaStream_t st, bool pdl, bool wait_tiles,
                           uint64_t budget_ns, bool gated) {
  const int n = d.R * d.H / 8;
  return launch_k(k_combine, dim3((n + 255) / 256), dim3(256), 0, st, pdl, d, s, out,
                  residual, wait_tiles, budget_ns, gated);
}

}  // namespace mtail
