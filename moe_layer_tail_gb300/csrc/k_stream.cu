// k_stream.cu -- the weight-streaming expert kernels: every distinct routed expert and the
// shared expert stream their weights from HBM exactly once per call.
//
// Work: the gate/up launch (PHASE 0) runs, for each group of 64 intermediate columns j,
// the 64 gate + 64 up weight rows of the shared expert (bf16) and of every distinct routed
// expert d (MXFP4) against every row that uses them.  The down launch (PHASE 1) runs, for
// each group of 128 hidden outputs, the 128 w2 rows of the shared expert and of every
// distinct routed expert against each user's SiLU*up vector.  A row's result never depends
// on which other rows share its expert: each output column of the contraction belongs to
// one user, and every sum runs in the same order whoever else is present.
//
// Sources: "[AMD] integrate kimi k3 monokernel" page, Kernel Replacement rows "The routed
// experts" and "The shared expert gate_up / SiLU and mul / down"; "glm53: Long-context
// indexer ..." page, Modifications rows 16 (each expert once in up/gate and down, every
// using row as a column of one multi-column product), 17 (no work for experts nobody
// picked), 18 (wide weight loads) and 21 (weights read once per call bypass the caches).
//
// Machine mapping (sm_103a), one CTA per SM, warp-specialised:
//   * warp 0, lane 0 -- the producer: takes items from a global atomic counter (shared-expert
//     items first, they are the largest) and, per pipeline stage, issues one or two 2D TMA
//     loads of a 128-row x 128-byte weight tile (128-byte swizzle, L2 evict-first) plus one
//     TMA load of the users' activation slice; every 8 stages of a routed item it adds the
//     E8M0 weight scales (and, for down, the activation block scales) of the next 2048 K
//     elements into a separate two-slot window ring.  Nothing but TMA issue and mbarrier
//     bookkeeping runs on this thread, so a stage costs it a few hundred cycles at most;
//   * warps 3..18 -- 16 consumer warps: warp c works on MMA tile m = c & 7 (16 weight rows)
//     and half h = c >> 3 of every stage's K range.  MXFP4 bytes go through
//     cvt.rn.f16x2.e2m1x2 straight into mma.m16n8k16 A fragments (weights = M rows, users =
//     N columns), each 32-element block's product is scaled by its E8M0 scale (times the
//     activation block scale for down) and accumulated in fp32; the shared expert is
//     bf16 x bf16 into fp32.  At the end of an item each warp drops its partial sums into a
//     reduction slot and moves on -- no consumer ever waits for another consumer;
//   * warps 1 and 2 -- the epilogue, taking items in turn: adds the two K halves of every
//     tile in a fixed order and finishes the item (SiLU*up, the f16 copy of mid with its
//     block scales, stores), then counts it done for its readers;
//   * activations enter the routed contractions as f16 with power-of-two scales (one per row
//     for gate/up, applied in the epilogue; for down, mid's 32-element blocks are unscaled
//     unless one falls outside f16's exact range, which switches that expert's down items to
//     per-block scales), exact for bf16 values in range;
//   * the two launches synchronise through counts, not grids: gate/up waits for the router
//     launch and then lets the down launch queue at once; down CTAs take the SMs gate/up
//     CTAs leave, and a down item's producer waits for the gate/up items it reads (counted
//     per distinct expert), so down overlaps the gate/up tail; down's epilogues count the
//     items of every 128 outputs for the combine;
//   * every wait is bounded by a %globaltimer budget; on expiry the kernel sets the status
//     word, lets the copies it issued land, and leaves.
#include <cstring>

#include "k_stream_common.cuh"

namespace mtail {

constexpr int kConsumerWarps = 16;
constexpr int kEpilogueWarps = 2;  // one per reduction slot
constexpr int kStreamThreads = (1 + kEpilogueWarps + kConsumerWarps) * 32;
constexpr int kActPitch = 512;    // routed activation rows: 256 f16 per stage

// --------------------------------------------------------------- shared-memory plan ----

struct SmemPtrs {
  uint8_t* stages;
  uint8_t* win;      // [2][win_bytes]
  float4* red;       // [2][16 warps][nt_max][32 lanes]
  int* t_uniq;
  int* t_off;
  int* t_users;
  float* t_rscale;
  uint64_t* full;    // [stages] producer -> consumers (transaction bytes)
  uint64_t* empty;   // [stages] consumers -> producer (16 arrivals)
  uint64_t* wempty;  // [2] consumers -> producer: scale window slot free
  uint64_t* rfull;   // [2] consumers -> epilogue: partial sums written (16 arrivals)
  uint64_t* rempty;  // [2] epilogue -> consumers: reduction slot read
  int2* info;        // [stages] item, k-chunk of each stage
  int* rinfo;        // [2] item of each reduction slot
};

__device__ __forceinline__ SmemPtrs carve_smem(uint8_t* smem, const StreamLayout& L) {
  SmemPtrs p;
  p.stages = smem;
  p.win = smem + L.off_win;
  p.red = reinterpret_cast<float4*>(smem + L.off_red);
  p.t_uniq = reinterpret_cast<int*>(smem + L.off_tab);
  p.t_off = p.t_uniq + L.tab_picks;
  p.t_users = p.t_off + L.tab_picks + 1;
  p.t_rscale = reinterpret_cast<float*>(p.t_users + L.tab_picks);
  p.full = reinterpret_cast<uint64_t*>(smem + L.off_bar);
  p.empty = p.full + kMaxStreamStages;
  p.wempty = p.empty + kMaxStreamStages;
  p.rfull = p.wempty + 2;
  p.rempty = p.rfull + 2;
  p.info = reinterpret_cast<int2*>(p.rempty + 2);
  p.rinfo = reinterpret_cast<int*>(p.info + kMaxStreamStages);
  return p;
}

// --------------------------------------------------------------------- consumers ----

// Per-lane shared-memory offsets fixed for the kernel: warp c works on MMA tile m = c & 7
// and on half h = c >> 3 of every stage's K range.
struct Lane {
  // routed (MXFP4): this lane's row address for the two ldmatrix.x4 loads of a stage; load
  // p returns word t of block chunks 4h + 2p and 4h + 2p + 1 of A rows a (MMA rows 0-7)
  // and b (8-15) as {a, b, a', b'}
  int ldsm[2];
  // routed: the rows' E8M0 bytes inside a scale window (add the block offset)
  int scale_a, scale_b;
  // shared (bf16): chunk 2t + h of A rows a and b
  int bw_a, bw_b;
};

__device__ __forceinline__ Lane make_lane(bool gate_up, int cw, int lane, int spitch) {
  Lane L;
  const int m = cw & 7, h = cw >> 3;
  const int g = lane >> 2, t = lane & 3;
  // A rows a and b of MMA row r (0-7): gate/up -- gate box rows 8m+r and up box rows 8m+r;
  // down -- one 128-row box, rows 16m+r and 16m+r+8
  const int abase = gate_up ? 8 * m : 16 * m;
  const int bbase = gate_up ? 8 * m : 16 * m + 8;
  const int boxb = gate_up ? 8192 : 0;
  const int sb0 = gate_up ? 4096 : 0;
  const int ra = abase + g, rb = bbase + g;
  {
    // ldmatrix: lane i addresses row i & 7 of matrix i >> 3 (a, b, a', b')
    const int j = lane >> 3, r = lane & 7;
    const int row = (j & 1) ? bbase + r : abase + r;
    const int box = (j & 1) ? boxb : 0;
#pragma unroll
    for (int p = 0; p < 2; ++p) L.ldsm[p] = box + swz128_off(row, 4 * h + 2 * p + (j >> 1));
  }
  L.scale_a = ra * spitch + 4 * h;
  L.scale_b = sb0 + rb * spitch + 4 * h;
  L.bw_a = swz128_off(ra, 2 * t + h);
  L.bw_b = boxb + swz128_off(rb, 2 * t + h);
  return L;
}

// Per-item offsets of this lane's users (N columns 8nt + g for the B fragments; columns
// 8nt + 2t and 8nt + 2t + 1 for the down activation scales).
struct UserOffs {
  int act[2];
  int as0[2], as1[2];
};

// One stage of a routed MXFP4 item: 4 scale blocks x 1 tile per warp.  Each block's two
// k16 products are scaled by the row's E8M0 scale (and, for down, the user's block scale)
// and added to the fp32 accumulators.  `sblk` = byte offset of this warp's first block in
// the window rows; `wsb` = the window slot.
template <bool GATE_UP, int NT, bool ACT_SCALED>
__device__ __forceinline__ void stage_routed(const uint8_t* st, const uint8_t* wsb,
                                             const Lane& L, const UserOffs& uo, int sblk,
                                             float (&acc)[2][4]) {
  const uint32_t swa = *reinterpret_cast<const uint32_t*>(wsb + L.scale_a + sblk);
  const uint32_t swb = *reinterpret_cast<const uint32_t*>(wsb + L.scale_b + sblk);
  float4 as0[NT], as1[NT];  // down: block scales of users (2t, 2t+1), per N-tile
  if (!GATE_UP && ACT_SCALED) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      as0[nt] = *reinterpret_cast<const float4*>(wsb + uo.as0[nt] + 4 * sblk);
      as1[nt] = *reinterpret_cast<const float4*>(wsb + uo.as1[nt] + 4 * sblk);
    }
  }
  uint32_t code[2][4];
#pragma unroll
  for (int p = 0; p < 2; ++p) ldsm_x4(st + L.ldsm[p], code[p]);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t wa = code[c >> 1][2 * (c & 1)];
    const uint32_t wb = code[c >> 1][2 * (c & 1) + 1];
    uint32_t ha[4], hb[4];
    e2m1x8_to_f16x2(wa, ha[0], ha[1], ha[2], ha[3]);
    e2m1x8_to_f16x2(wb, hb[0], hb[1], hb[2], hb[3]);
    const float sa = e8m0_byte(swa, c), sb = e8m0_byte(swb, c);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const uint4 b = *reinterpret_cast<const uint4*>(st + uo.act[nt] + c * 64);
      float tmp[4];
      mma_f16_z(tmp, ha[0], hb[0], ha[1], hb[1], b.x, b.y);
      mma_f16(tmp, ha[2], hb[2], ha[3], hb[3], b.z, b.w);
      if (GATE_UP || !ACT_SCALED) {
        acc[nt][0] += tmp[0] * sa;
        acc[nt][1] += tmp[1] * sa;
        acc[nt][2] += tmp[2] * sb;
        acc[nt][3] += tmp[3] * sb;
      } else {
        const float u0 = (c == 0) ? as0[nt].x : (c == 1) ? as0[nt].y : (c == 2) ? as0[nt].z : as0[nt].w;
        const float u1 = (c == 0) ? as1[nt].x : (c == 1) ? as1[nt].y : (c == 2) ? as1[nt].z : as1[nt].w;
        acc[nt][0] += tmp[0] * (sa * u0);
        acc[nt][1] += tmp[1] * (sa * u1);
        acc[nt][2] += tmp[2] * (sb * u0);
        acc[nt][3] += tmp[3] * (sb * u1);
      }
    }
  }
}

// One stage of a shared-expert (bf16) item: 32 K elements (half h) x 1 tile per warp.
// Lane t takes elements [16t + 8h, +8) of the 64-element stage row, for its two A rows and
// for user g (conflict-free under the 128-byte swizzle).
template <int NT>
__device__ __forceinline__ void stage_shared(const uint8_t* st, const Lane& L,
                                             const UserOffs& uo, float (&acc)[2][4]) {
  const uint4 a = *reinterpret_cast<const uint4*>(st + L.bw_a);
  const uint4 c = *reinterpret_cast<const uint4*>(st + L.bw_b);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const uint4 b = *reinterpret_cast<const uint4*>(st + uo.act[nt]);
    mma_bf16(acc[nt], a.x, c.x, a.y, c.y, b.x, b.y);
    mma_bf16(acc[nt], a.z, c.z, a.w, c.w, b.z, b.w);
  }
}

// The ring position of a consumer warp: stage slot, its phase parity, scale windows seen.
struct Ring {
  int stage;
  uint32_t phase, wcnt;
};

// All stages of one item for one consumer warp; the item's first stage has already been
// waited for.  Returns false when a wait ran out of budget.
template <bool GATE_UP, int NT, bool ACT_SCALED>
__device__ __forceinline__ bool run_routed(const SmemPtrs& sp, const StreamLayout& lay, Ring& rg,
                                        const Item& it, const Lane& L, const UserOffs& uo,
                                        int eh, uint64_t budget_ns, float (&acc)[2][4]) {
  const int lane = threadIdx.x & 31;
  const uint8_t* wsb = sp.win + (rg.wcnt & 1u) * lay.win_bytes;
  // this warp's half of the last stage may lie past K
  const bool last_has_k = (it.nst - 1) * kChunkF4 + (kChunkF4 / 2) * eh < it.K;
  for (int kc = 0; kc < it.nst; ++kc) {
    if (kc > 0 && !mbar_wait(&sp.full[rg.stage], rg.phase, budget_ns)) return false;
    if (kc < it.nst - 1 || last_has_k)
      stage_routed<GATE_UP, NT, ACT_SCALED>(sp.stages + rg.stage * lay.stage_bytes, wsb, L, uo,
                                (kc % kWinStages) * 8, acc);
    __syncwarp();
    if (lane == 0) mbar_arrive(&sp.empty[rg.stage]);
    if (++rg.stage == lay.stages) { rg.stage = 0; rg.phase ^= 1; }
    if ((kc % kWinStages) == kWinStages - 1 || kc == it.nst - 1) {
      if (lane == 0) mbar_arrive(&sp.wempty[rg.wcnt & 1u]);
      ++rg.wcnt;
      wsb = sp.win + (rg.wcnt & 1u) * lay.win_bytes;
    }
  }
  return true;
}

template <int NT>
__device__ __forceinline__ bool run_shared(const SmemPtrs& sp, const StreamLayout& lay, Ring& rg,
                                        const Item& it, const Lane& L, const UserOffs& uo,
                                        int eh, uint64_t budget_ns, float (&acc)[2][4]) {
  const int lane = threadIdx.x & 31;
  const bool last_has_k = (it.nst - 1) * kChunkBF + (kChunkBF / 2) * eh < it.K;
  for (int kc = 0; kc < it.nst; ++kc) {
    if (kc > 0 && !mbar_wait(&sp.full[rg.stage], rg.phase, budget_ns)) return false;
    if (kc < it.nst - 1 || last_has_k)
      stage_shared<NT>(sp.stages + rg.stage * lay.stage_bytes, L, uo, acc);
    __syncwarp();
    if (lane == 0) mbar_arrive(&sp.empty[rg.stage]);
    if (++rg.stage == lay.stages) { rg.stage = 0; rg.phase ^= 1; }
  }
  return true;
}

// --------------------------------------------------------------------- epilogue ----

// Tile m's sums for N-tile nt: (half 0) + (half 1), in that order.
__device__ __forceinline__ void tile_sum(const float4* rb, int nt_max, int m, int nt, int lane,
                                         float (&c)[4]) {
  const float4 v0 = rb[(m * nt_max + nt) * 32 + lane];
  const float4 v1 = rb[((m + 8) * nt_max + nt) * 32 + lane];
  c[0] = v0.x + v1.x;
  c[1] = v0.y + v1.y;
  c[2] = v0.z + v1.z;
  c[3] = v0.w + v1.w;
}

__device__ __forceinline__ void finish_item(const Item& it, const float4* rb, int nt_max,
                                         const Dims& dm, const Tables& tb, const Scratch& s,
                                         int lane) {
  const int g = lane >> 2, t = lane & 3;
  const int NT = it.U > 8 ? 2 : 1;
  for (int nt = 0; nt < NT; ++nt) {
    if (it.kind == kSharedGU) {
      for (int m = 0; m < 8; ++m) {
        float c[4];
        tile_sum(rb, nt_max, m, nt, lane, c);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int r = nt * 8 + 2 * t + q;
          if (r < it.U)
            s.ms[(size_t)r * dm.Is + it.out0 + 8 * m + g] =
                __float2bfloat16_rn(silu_f(c[q]) * c[2 + q]);
        }
      }
    } else if (it.kind == kOutProj) {
      // rows 16m + g and 16m + g + 8 of the 128-output box: x = bf16(attn . W_o^T) when the
      // box is one part, else this part's fp32 sums (the norm launch adds the parts in order)
      for (int m = 0; m < 8; ++m) {
        float c[4];
        tile_sum(rb, nt_max, m, nt, lane, c);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int u = nt * 8 + 2 * t + q;
          if (u < it.U) {
            if (dm.Pk == 1) {
              __nv_bfloat16* xr = s.xproj + (size_t)u * dm.H + it.out0;
              xr[16 * m + g] = __float2bfloat16_rn(c[q]);
              xr[16 * m + g + 8] = __float2bfloat16_rn(c[2 + q]);
            } else {
              float* xr = s.xpart + ((size_t)it.part * dm.Rmax + u) * dm.H + it.out0;
              xr[16 * m + g] = c[q];
              xr[16 * m + g + 8] = c[2 + q];
            }
          }
        }
      }
    } else if (it.kind == kSharedDN || it.kind == kRoutedDN) {
      float* rows[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int u = nt * 8 + 2 * t + q;
        rows[q] = nullptr;
        if (u < it.U)
          rows[q] = (it.kind == kSharedDN) ? s.ys + (size_t)u * dm.H + it.out0
                                           : s.y + (size_t)tb.users[it.u0 + u] * dm.H + it.out0;
      }
      for (int m = 0; m < 8; ++m) {
        float c[4];
        tile_sum(rb, nt_max, m, nt, lane, c);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          if (rows[q] != nullptr) {
            rows[q][16 * m + g] = c[q];
            rows[q][16 * m + g + 8] = c[2 + q];
          }
        }
      }
    } else {
      // routed gate/up: mid = bf16(SiLU(gate) * up) with the row's activation scale
      // restored; its f16 copy gets one power-of-two scale per (user, 32 columns)
      float rs[2];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int u = nt * 8 + 2 * t + q;
        rs[q] = (u < it.U) ? tb.rscale[tb.users[it.u0 + u] / dm.k] : 0.f;
      }
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float mv[4][2];
        float amax[2] = {0.f, 0.f};
#pragma unroll
        for (int mm = 0; mm < 4; ++mm) {
          float c[4];
          tile_sum(rb, nt_max, 4 * half + mm, nt, lane, c);
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            mv[mm][q] = __bfloat162float(
                __float2bfloat16_rn(silu_f(c[q] * rs[q]) * (c[2 + q] * rs[q])));
            amax[q] = fmaxf(amax[q], fabsf(mv[mm][q]));
          }
        }
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          amax[q] = fmaxf(amax[q], __shfl_xor_sync(0xffffffffu, amax[q], 4));
          amax[q] = fmaxf(amax[q], __shfl_xor_sync(0xffffffffu, amax[q], 8));
          amax[q] = fmaxf(amax[q], __shfl_xor_sync(0xffffffffu, amax[q], 16));
          const int u = nt * 8 + 2 * t + q;
          if (u < it.U) {
            // blocks whose largest magnitude lies in [2^-10, 2^15) are stored unscaled: f16
            // holds their bf16 values exactly down to 2^-14 and the smaller ones within 2^-25;
            // any other block gets a power of two and marks the call as scaled
            int p = 0;
            if (amax[q] > 0.f) {
              const int ex = (int)((__float_as_uint(amax[q]) >> 23) & 0xFF) - 127;
              if (ex < -10 || ex > 14) {
                p = max(-100, min(100, ex - 14));
                if (g == 0) atomicOr(&s.counters[kCtrMidFlag + it.d], 1u);
              }
            }
            const float down = __uint_as_float((uint32_t)(127 - p) << 23);
            const size_t slot = (size_t)(it.u0 + u);
            __half* mrow = s.mid16 + slot * dm.I + it.out0 + 32 * half;
#pragma unroll
            for (int mm = 0; mm < 4; ++mm) mrow[8 * mm + g] = __float2half_rn(mv[mm][q] * down);
            if (g == 0)
              s.mid16s[slot * (dm.I / 32) + it.out0 / 32 + half] =
                  __uint_as_float((uint32_t)(127 + p) << 23);
          }
        }
      }
    }
  }
}

// ------------------------------------------------------------------------ kernel ----


template <int PHASE>
__global__ void __launch_bounds__(kStreamThreads, 1)
k_stream(const __grid_constant__ StreamMaps maps, Dims dm, Weights w, Scratch s,
         uint64_t budget_ns, uint32_t debug) {
  // The dynamic shared memory starts 1024-byte aligned (nothing else is in shared memory),
  // as the swizzled TMA boxes need; every pointer below stays in the shared space.
  extern __shared__ __align__(1024) uint8_t smem[];
  const StreamLayout& lay = maps.lay;
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) set_status(s.status, kStatusBadTile);
    return;
  }
  const SmemPtrs sp = carve_smem(smem, lay);
  const int S = lay.stages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Gate/up waits for the routing.  Down does not wait for the gate/up grid as a whole: it is
  // launched once every gate/up CTA has passed that wait (so the routing is complete), its
  // CTAs take the SMs the gate/up CTAs leave, and each down item waits, in its producer,
  // for the gate/up items whose output it reads (counted by their epilogues).
  if (PHASE != 1) pdl_wait();
  const int D = min(max(*s.n_distinct, 1), kMaxPicks);
  const int n_items = items_of(PHASE, dm, D);
  for (int i = threadIdx.x; i < D; i += kStreamThreads) sp.t_uniq[i] = s.uniq[i];
  for (int i = threadIdx.x; i <= D; i += kStreamThreads) sp.t_off[i] = s.user_off[i];
  for (int i = threadIdx.x; i < dm.R * dm.k; i += kStreamThreads) sp.t_users[i] = s.user_list[i];
  for (int i = threadIdx.x; i < dm.R; i += kStreamThreads) sp.t_rscale[i] = s.n16s[i];
  Tables tb;
  tb.uniq = sp.t_uniq;
  tb.off = sp.t_off;
  tb.users = sp.t_users;
  tb.rscale = sp.t_rscale;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&sp.full[i], 1);
      mbar_init(&sp.empty[i], kConsumerWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sp.wempty[i], kConsumerWarps);
      mbar_init(&sp.rfull[i], kConsumerWarps);
      mbar_init(&sp.rempty[i], 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    pdl_trigger();  // the next launch may queue for SMs from now on (it waits on counts)
  }
  __syncthreads();

  // K length of the routed contraction and the byte pitch of its scale-window rows
  const int Kr = (PHASE == 0) ? dm.H : dm.I;
  const int spitch = (Kr > kWinK) ? 64 : Kr / 32;
  const int apitch = 4 * min(64, dm.I / 32);  // down: activation-scale window rows

  if (warp == 0) {
    // ---------------------------------------------------------------- producer ----
    if (lane != 0) return;
    const uint64_t pol = policy_evict_first();
    int stage = 0;
    uint32_t phase = 0;
    uint32_t wcnt = 0;  // scale windows issued so far
    bool ok = true;
    // stages whose copies were issued and not yet seen consumed, with their phase parity
    uint32_t pend = 0u, pend_par = 0u;
    // failure-injection switch: CTA 0 leaves its first stage unpublished, so the consumers'
    // bounded wait on it expires (tests the timeout path; never set in production)
    bool skip_first = PHASE == 0 && (debug & kDebugStallFirstStage) && blockIdx.x == 0;
    int item = (int)atomicAdd(&s.counters[work_counter(PHASE)], 1u);
    while (ok && item < n_items) {
      const int next = (int)atomicAdd(&s.counters[work_counter(PHASE)], 1u);  // lands while this streams
      const Item it = decode_item(PHASE, item, dm, tb, D);
      const bool routed = (it.kind == kRoutedGU || it.kind == kRoutedDN);
      const int hsel = (it.U <= 4) ? 0 : (it.U <= 8) ? 1 : 2;  // down activation box height
      int scaled = 0;  // routed down: some block of the expert's mid carries a scale
      if (PHASE == 1) {
        // the gate/up items this one reads must be finished (their epilogues' stores made
        // visible to this thread, then to the copy engine)
        const bool sh = (it.kind == kSharedDN);
        if (!wait_count(&s.counters[sh ? kCtrSharedGUDone : kCtrGUDone + it.d],
                        (uint32_t)(sh ? dm.Is / 64 : dm.I / 64), budget_ns)) {
          ok = false;
          break;
        }
        asm volatile("fence.proxy.async.global;" ::: "memory");
        if (!sh) scaled = *(volatile const uint32_t*)&s.counters[kCtrMidFlag + it.d] != 0u;
      }
      uint32_t act_bytes;
      if (it.kind == kRoutedGU) act_bytes = (uint32_t)dm.Rmax * kActPitch;
      else if (it.kind == kRoutedDN) act_bytes = (4u << hsel) * kActPitch;
      else act_bytes = (uint32_t)dm.Rmax * 128u;
      for (int kc = 0; kc < it.nst; ++kc) {
        if (!mbar_wait(&sp.empty[stage], phase ^ 1, budget_ns)) { ok = false; break; }
        pend &= ~(1u << stage);
        if (skip_first) {
          skip_first = false;
          if (++stage == S) { stage = 0; phase ^= 1; }
          continue;
        }
        uint8_t* st = sp.stages + stage * lay.stage_bytes;
        uint32_t bytes = kStageW + act_bytes;
        const bool wstart = routed && (kc % kWinStages) == 0;
        uint8_t* ws = sp.win + (wcnt & 1u) * lay.win_bytes;
        uint32_t wbytes = 0;
        if (wstart) {
          if (!mbar_wait(&sp.wempty[wcnt & 1u], ((wcnt >> 1) & 1u) ^ 1u, budget_ns)) {
            ok = false;
            break;
          }
          if (PHASE == 0) wbytes = (Kr > kWinK) ? 8192u : 4u * (uint32_t)Kr;
          else wbytes = ((Kr > kWinK) ? 8192u : 4u * (uint32_t)Kr) + (4u << hsel) * (uint32_t)apitch;
          bytes += wbytes;
        }
        pend |= 1u << stage;
        pend_par = (pend_par & ~(1u << stage)) | (phase << stage);
        sp.info[stage] = make_int2(item, scaled);
        mbar_expect_tx(&sp.full[stage], bytes);
        uint8_t* sa = st + kStageW;
        if (it.kind == kRoutedGU) {
          const int x = kc * (kChunkF4 / 2);
          tma_load_2d(st, &maps.w13, x, it.row0, &sp.full[stage], pol);
          tma_load_2d(st + 8192, &maps.w13, x, it.row1, &sp.full[stage], pol);
          tma_load_2d(sa, &maps.n16, kc * kChunkF4, 0, &sp.full[stage]);
        } else if (it.kind == kRoutedDN) {
          tma_load_2d(st, &maps.w2, kc * (kChunkF4 / 2), it.row0, &sp.full[stage], pol);
          tma_load_2d(sa, &maps.mid16[hsel], kc * kChunkF4, it.u0, &sp.full[stage]);
        } else if (it.kind == kOutProj) {
          const int x = it.k0 + kc * kChunkBF;
          tma_load_2d(st, &maps.wo, x, it.row0, &sp.full[stage], pol);
          tma_load_2d(sa, &maps.attn, x, 0, &sp.full[stage]);
        } else if (it.kind == kSharedGU) {
          tma_load_2d(st, &maps.ws13, kc * kChunkBF, it.row0, &sp.full[stage], pol);
          tma_load_2d(st + 8192, &maps.ws13, kc * kChunkBF, it.row1, &sp.full[stage], pol);
          tma_load_2d(sa, &maps.n, kc * kChunkBF, 0, &sp.full[stage]);
        } else {
          tma_load_2d(st, &maps.ws2, kc * kChunkBF, it.row0, &sp.full[stage], pol);
          tma_load_2d(sa, &maps.ms, kc * kChunkBF, 0, &sp.full[stage]);
        }
        if (wstart) {
          const int win = kc / kWinStages;
          if (PHASE == 0) {
            if (Kr > kWinK) {
              tma_load_2d(ws, &maps.w13s, win * 64, it.row0, &sp.full[stage]);
              tma_load_2d(ws + 4096, &maps.w13s, win * 64, it.row1, &sp.full[stage]);
            } else {  // the whole K of the 64 gate and 64 up rows: two contiguous runs
              const size_t rb = (size_t)(Kr / 32);
              bulk_load(ws, w.w13s + (size_t)it.row0 * rb, 2u * (uint32_t)Kr, &sp.full[stage]);
              bulk_load(ws + 4096, w.w13s + (size_t)it.row1 * rb, 2u * (uint32_t)Kr,
                        &sp.full[stage]);
            }
          } else {
            if (Kr > kWinK) {
              tma_load_2d(ws, &maps.w2s, win * 64, it.row0, &sp.full[stage]);
            } else {
              const size_t rb = (size_t)(Kr / 32);
              bulk_load(ws, w.w2s + (size_t)it.row0 * rb, 4u * (uint32_t)Kr, &sp.full[stage]);
            }
            tma_load_2d(ws + kWinW, &maps.mid16s[hsel], win * 64, it.u0, &sp.full[stage]);
          }
          ++wcnt;
        }
        if (++stage == S) { stage = 0; phase ^= 1; }
      }
      item = next;
    }
    if (ok) {
      // end-of-work marker (withheld too by the failure injection, when this CTA got no
      // item to stall on)
      ok = mbar_wait(&sp.empty[stage], phase ^ 1, budget_ns);
      if (ok && !skip_first) {
        sp.info[stage] = make_int2(-1, 0);
        mbar_arrive(&sp.full[stage]);
      }
    }
    if (!ok) {
      // a wait expired: record it, then let every copy this CTA issued land (bounded)
      // before the CTA's shared memory is released
      set_status(s.status, kStatusTimeout);
      for (int st2 = 0; st2 < S; ++st2)
        if (pend & (1u << st2)) mbar_wait(&sp.full[st2], (pend_par >> st2) & 1u, budget_ns);
    }
    return;
  }

  if (warp <= kEpilogueWarps) {
    // ---------------------------------------------------------------- epilogue ----
    // epilogue warp w finishes the items of reduction slot w - 1 (every other item)
    for (uint32_t rc = (uint32_t)(warp - 1);; rc += kEpilogueWarps) {
      const uint32_t rb = rc & 1u;
      if (!mbar_wait(&sp.rfull[rb], (rc >> 1) & 1u, budget_ns)) {
        if (lane == 0) set_status(s.status, kStatusTimeout);
        break;
      }
      const int item = sp.rinfo[rb];
      if (item < 0) break;
      const Item it = decode_item(PHASE, item, dm, tb, D);
      finish_item(it, sp.red + rb * (kConsumerWarps * lay.nt_max * 32), lay.nt_max, dm, tb, s,
                  lane);
      // count the item for its readers (the down items of the expert, or the combine of its
      // 128 outputs): the warp barrier orders every lane's stores before lane 0's release
      __syncwarp();
      if (PHASE != 2 && lane == 0) {  // (the norm launch waits for out_proj as a whole)
        uint32_t* c = &s.counters[PHASE == 1 ? kCtrTileDone + it.out0 / 128
                                  : it.kind == kSharedGU ? kCtrSharedGUDone
                                                         : kCtrGUDone + it.d];
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(c) : "memory");
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sp.rempty[rb]);
    }
    return;
  }

  // ------------------------------------------------------------------ consumers ----
  const int cw = warp - 1 - kEpilogueWarps;
  const int g = lane >> 2, t = lane & 3;
  const int eh = cw >> 3;  // this warp's K half
  const Lane L = make_lane(PHASE == 0, cw, lane, spitch);
  Ring rg;
  rg.stage = 0;
  rg.phase = 0;
  rg.wcnt = 0;
  uint32_t rc = 0;
  bool ok = true;
  for (;;) {
    if (!mbar_wait(&sp.full[rg.stage], rg.phase, budget_ns)) { ok = false; break; }
    const int2 info = sp.info[rg.stage];
    const int item = info.x;
    if (item < 0) {
      // end of work: hand each epilogue warp the end marker through its next reduction slot
      for (int q = 0; q < kEpilogueWarps && ok; ++q, ++rc) {
        const uint32_t rb = rc & 1u;
        if (mbar_wait(&sp.rempty[rb], ((rc >> 1) & 1u) ^ 1u, budget_ns)) {
          if (cw == 0 && lane == 0) sp.rinfo[rb] = -1;
          __syncwarp();
          if (lane == 0) mbar_arrive(&sp.rfull[rb]);
        } else {
          ok = false;
        }
      }
      break;
    }
    const Item it = decode_item(PHASE, item, dm, tb, D);
    const int NT = it.U > 8 ? 2 : 1;
    UserOffs uo;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int n = min(nt * 8 + g, it.U - 1);  // B column of this lane (clamped)
      if (it.kind == kRoutedGU)
        uo.act[nt] = kStageW + (tb.users[it.u0 + n] / dm.k) * kActPitch + eh * 256 + 16 * t;
      else if (it.kind == kRoutedDN)
        uo.act[nt] = kStageW + n * kActPitch + eh * 256 + 16 * t;
      else
        uo.act[nt] = kStageW + swz128_off(n, 2 * t + eh);
      const int u0c = min(nt * 8 + 2 * t, it.U - 1), u1c = min(nt * 8 + 2 * t + 1, it.U - 1);
      uo.as0[nt] = kWinW + u0c * apitch + 16 * eh;
      uo.as1[nt] = kWinW + u1c * apitch + 16 * eh;
    }
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    if (it.kind == kRoutedGU || it.kind == kRoutedDN) {
      if (PHASE == 0 || info.y == 0)
        ok = (NT == 1) ? run_routed<PHASE == 0, 1, false>(sp, lay, rg, it, L, uo, eh, budget_ns, acc)
                       : run_routed<PHASE == 0, 2, false>(sp, lay, rg, it, L, uo, eh, budget_ns, acc);
      else
        ok = (NT == 1) ? run_routed<false, 1, true>(sp, lay, rg, it, L, uo, eh, budget_ns, acc)
                       : run_routed<false, 2, true>(sp, lay, rg, it, L, uo, eh, budget_ns, acc);
    } else {
      ok = (NT == 1) ? run_shared<1>(sp, lay, rg, it, L, uo, eh, budget_ns, acc)
                     : run_shared<2>(sp, lay, rg, it, L, uo, eh, budget_ns, acc);
    }
    if (!ok) break;
    // item end: partial sums to the next reduction slot, then on to the next item
    const uint32_t rb = rc & 1u;
    if (!mbar_wait(&sp.rempty[rb], ((rc >> 1) & 1u) ^ 1u, budget_ns)) { ok = false; break; }
    float4* red = sp.red + rb * (kConsumerWarps * lay.nt_max * 32);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
      if (nt < NT)
        red[(cw * lay.nt_max + nt) * 32 + lane] =
            make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
    if (cw == 0 && lane == 0) sp.rinfo[rb] = item;
    __syncwarp();
    if (lane == 0) mbar_arrive(&sp.rfull[rb]);
    ++rc;
  }
  if (!ok && lane == 0) set_status(s.status, kStatusTimeout);
}

// Opt the streaming kernels in to the largest shared-memory size (once per process and
// device before the first launch; called at create time, outside any graph capture).
cudaError_t prepare_stream_kernels() {
  cudaError_t e = cudaFuncSetAttribute(k_stream<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemLimit);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_stream<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemLimit);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_stream<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kSmemLimit);
  return e;
}

cudaError_t launch_stream(int phase, const StreamMaps& maps, const Dims& d, const Weights& w,
                          const Scratch& s, int num_sms, uint64_t budget_ns, cudaStream_t st,
                          bool pdl, uint32_t debug) {
  const size_t smem = (size_t)maps.lay.smem_bytes;
  if (phase == 0)
    return launch_k(k_stream<0>, dim3(num_sms), dim3(kStreamThreads), smem, st, pdl, maps, d, w,
                    s, budget_ns, debug);
  if (phase == 1)
    return launch_k(k_stream<1>, dim3(num_sms), dim3(kStreamThreads), smem, st, pdl, maps, d,
                    w, s, budget_ns, debug);
  // out_proj: (H / 128) x Pk items, one CTA per item up to one per SM
  const int items = d.H / 128 * d.Pk;
  const int grid = items < num_sms ? items : num_sms;
  return launch_k(k_stream<2>, dim3(grid), dim3(kStreamThreads), smem, st, pdl, maps, d, w, s,
                  budget_ns, debug);
}

// ----------------------------------------------------------- tensor-map encoding ----

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static int encode_2d(EncodeTiledFn fn, CUtensorMap* m, CUtensorMapDataType dt, const void* base,
                     uint64_t inner, uint64_t rows, uint64_t row_bytes, uint32_t box_inner,
                     uint32_t box_rows, CUtensorMapSwizzle swz) {
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -1;
}

// Shared-memory plan for a handle created for `Rmax` rows (stages as many as fit, up to 8).
StreamLayout make_stream_layout(int Rmax, int k) {
  StreamLayout L;
  L.tab_picks = Rmax * k;
  L.act_rows = (Rmax <= 4) ? 4 : (Rmax <= 8) ? 8 : 16;
  L.stage_bytes = kStageW + L.act_rows * kActPitch;
  L.win_bytes = kWinW + L.act_rows * 256;
  L.nt_max = (Rmax > 8) ? 2 : 1;
  const int red_bytes = 2 * kConsumerWarps * L.nt_max * 512;
  const int tab_bytes = ((3 * L.tab_picks + 1 + Rmax) * 4 + 127) & ~127;
  const int bar_bytes = (2 * kMaxStreamStages + 6) * 8 + kMaxStreamStages * 8 + 2 * 4;
  const int fixed = 2 * L.win_bytes + red_bytes + tab_bytes + ((bar_bytes + 127) & ~127);
  L.stages = min(kMaxStreamStages, (kSmemLimit - fixed) / L.stage_bytes);
  L.off_win = L.stages * L.stage_bytes;
  L.off_red = L.off_win + 2 * L.win_bytes;
  L.off_tab = L.off_red + red_bytes;
  L.off_bar = L.off_tab + tab_bytes;
  L.smem_bytes = L.off_bar + ((bar_bytes + 127) & ~127);
  return L;
}

// Every weight box has 128-byte rows (the 128-byte swizzle span): 128 MXFP4 code bytes (256
// elements) or 64 bf16 elements.  Returns 0 on success, -1 if the driver has no tensor-map
// encoder, -2 if encoding failed.
static EncodeTiledFn tensor_map_encoder() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess)
      fn = (EncodeTiledFn)p;
  }
  return fn;
}

int make_attn_map(StreamMaps* m, const void* attn, int rows, const Dims& d) {
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return -1;
  // rows past the call's are filled with zeros by the copy engine (their outputs unused)
  if (encode_2d(enc, &m->attn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, attn, (uint64_t)d.Ha,
                (uint64_t)rows, (uint64_t)d.Ha * 2, 64, (uint32_t)d.Rmax,
                CU_TENSOR_MAP_SWIZZLE_128B))
    return -2;
  return 0;
}

int make_stream_maps(StreamMaps* out, const Dims& d, const Weights& w, const Scratch& s) {
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return -1;
  const uint64_t H = d.H, E = d.E, I = d.I, Is = d.Is, R = d.Rmax, P = (uint64_t)d.Rmax * d.k;
  const CUtensorMapDataType U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const CUtensorMapDataType BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapDataType F16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUtensorMapDataType F32 = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  const CUtensorMapSwizzle SW = CU_TENSOR_MAP_SWIZZLE_128B, NS = CU_TENSOR_MAP_SWIZZLE_NONE;
  memset(out, 0, sizeof(*out));
  if (encode_2d(enc, &out->w13, U8, w.w13c, H / 2, E * 2 * I, H / 2, 128, 64, SW)) return -2;
  if (encode_2d(enc, &out->w2, U8, w.w2c, I / 2, E * H, I / 2, 128, 128, SW)) return -2;
  if (encode_2d(enc, &out->ws13, BF, w.ws13, H, 2 * Is, H * 2, 64, 64, SW)) return -2;
  if (encode_2d(enc, &out->ws2, BF, w.ws2, Is, H, Is * 2, 64, 128, SW)) return -2;
  if (encode_2d(enc, &out->n, BF, s.n, H, R, H * 2, 64, (uint32_t)R, SW)) return -2;
  if (encode_2d(enc, &out->ms, BF, s.ms, Is, R, Is * 2, 64, (uint32_t)R, SW)) return -2;
  if (encode_2d(enc, &out->n16, F16, s.n16, H, R, H * 2, 256, (uint32_t)R, NS)) return -2;
  for (int i = 0; i < 3; ++i) {
    const uint32_t rows = 4u << i;
    if (encode_2d(enc, &out->mid16[i], F16, s.mid16, I, P, I * 2, 256, rows, NS)) return -2;
    if (encode_2d(enc, &out->mid16s[i], F32, s.mid16s, I / 32, P, (I / 32) * 4,
                  (uint32_t)(I / 32 < 64 ? I / 32 : 64), rows, NS))
      return -2;
  }
  // scale windows of 64 bytes per row, only where a row holds more than one window
  if (H > (uint64_t)kWinK &&
      encode_2d(enc, &out->w13s, U8, w.w13s, H / 32, E * 2 * I, H / 32, 64, 64, NS))
    return -2;
  if (I > (uint64_t)kWinK &&
      encode_2d(enc, &out->w2s, U8, w.w2s, I / 32, E * H, I / 32, 64, 128, NS))
    return -2;
  if (d.Ha > 0 &&
      encode_2d(enc, &out->wo, BF, w.wo, (uint64_t)d.Ha, H, (uint64_t)d.Ha * 2, 64, 128, SW))
    return -2;
  out->lay = make_stream_layout(d.Rmax, d.k);
  return 0;
}

// Tensor maps of the tensor-core streaming kernels: the weight and bf16 activation maps of
// the CUDA-core form, plus the E2M1 planes of n and mid (their scales, like the weights',
// travel as scale-factor atoms by plain bulk copies).  Returns 0,
// -1 (no encoder) or -2 (encoding failed).
int make_tc_maps(TcMaps* out, const StreamMaps& sm, const Dims& d, const Weights& w,
                 const Scratch& s, int smem_limit) {
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return -1;
  memset(out, 0, sizeof(*out));
  out->w2 = sm.w2;
  out->ws2 = sm.ws2;
  out->n = sm.n;
  out->ms = sm.ms;
  out->lay = make_tc_layout(d.Rmax, d.k, smem_limit);
  const uint32_t nmax = (uint32_t)out->lay.nmax;
  const uint64_t H = d.H, I = d.I, R4 = 4ull * d.Rmax, P4 = 4ull * d.Rmax * d.k;
  const CUtensorMapDataType U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const CUtensorMapSwizzle SW = CU_TENSOR_MAP_SWIZZLE_128B;
  {
    // gate and up rows of a stage in one 3-D box each: w13 as [2E][I][H/2] bytes, the shared
    // expert's ws13 as [2][Is][H] bf16
    cuuint64_t dims[3] = {H / 2, I, 2ull * d.E};
    cuuint64_t strides[2] = {H / 2, I * (H / 2)};
    cuuint32_t box[3] = {128, 64, 2};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&out->w13, U8, 3, const_cast<uint8_t*>(w.w13c), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, SW, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return -2;
    const uint64_t Is = d.Is;
    cuuint64_t dims2[3] = {H, Is, 2};
    cuuint64_t strides2[2] = {H * 2, Is * H * 2};
    cuuint32_t box2[3] = {64, 64, 2};
    if (enc(&out->ws13, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<__nv_bfloat16*>(w.ws13),
            dims2, strides2, box2, es, CU_TENSOR_MAP_INTERLEAVE_NONE, SW,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return -2;
  }
  // rows past 4 Rmax (planes) and 4 P (mid planes) read as zeros
  if (encode_2d(enc, &out->np4, U8, s.np4, H / 2, R4, H / 2, 128, nmax, SW)) return -2;
  for (int i = 0; i < 4; ++i) {
    const uint32_t rows = 16u << i;
    if (rows > nmax) break;
    if (encode_2d(enc, &out->mid4[i], U8, s.mid4, I / 2, P4, I / 2, 128, rows, SW)) return -2;
  }
  return 0;
}

}  // namespace mtail
