// k_combine.cuh -- the combine of one call, shared by the combine launch (k_simple.cu) and
// the single persistent launch (k_stream_tc.cu).
//
// out[r, h] = bf16(sum over slots in pick order of wts * y + ys): a fixed-order fp32 sum (the
// shared expert's term times its row's sigmoid gate when the layer has one); the residual
// receives bf16(x + residual), now that every reader of the old value is done.
// Source: "[AMD] integrate kimi k3 monokernel" page, Kernel checks table (out, res_out).
#pragma once

#include "moe_tail_internal.cuh"

namespace mtail {

// One thread's 8 outputs: row r, outputs 8c .. 8c + 7 (the slots' loads unrolled so that
// they are in flight together).
__device__ __forceinline__ void combine_one(const Dims& dm, const Scratch& s, int r, int c,
                                            __nv_bfloat16* __restrict__ out,
                                            __nv_bfloat16* __restrict__ residual, bool gated) {
  const int H = dm.H, k = dm.k;
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

// Wait (bounded, acquire) until the down items of the two 128-output tiles a warp's 256
// outputs cover (the shared expert's and one per distinct expert) are counted done; lanes 0
// and 16 wait, the others are ordered after them.  c: the lane's group of 8 outputs.  False
// (status set by lane 0) when a wait expired.  Whole warps only.
__device__ __forceinline__ bool combine_wait_tiles(const Scratch& s, int c, uint64_t budget_ns) {
  const int lane = threadIdx.x & 31;
  const uint32_t need = (uint32_t)min(max(__ldcg(s.n_distinct), 1), kMaxPicks) + 1u;
  bool ok = true;
  if ((lane & 15) == 0) ok = wait_count(&s.counters[kCtrTileDone + c / 16], need, budget_ns);
  if (__any_sync(0xffffffffu, !ok)) {
    if (lane == 0) set_status(s.status, kStatusTimeout);
    return false;
  }
  __syncwarp();
  return true;
}

// After a CTA's combine: when `done` is given, the last of the launch's nctas CTAs (a ticket
// after a system-scope fence in every CTA) writes seq to the host-visible word done with a
// system-scope release, so that a host thread that reads seq there (acquire) sees every
// output of the call.  Every thread of the CTA calls it.
__device__ __forceinline__ void signal_done(const Scratch& s, uint32_t* done, uint32_t seq,
                                            uint32_t nctas) {
  if (!done) return;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence_system();
    if (atomicAdd(&s.counters[kCtrCombineTicket], 1u) == nctas - 1u) {
      __threadfence_system();
      asm volatile("st.release.sys.global.u32 [%0], %1;" ::"l"(done), "r"(seq) : "memory");
    }
  }
}

}  // namespace mtail
