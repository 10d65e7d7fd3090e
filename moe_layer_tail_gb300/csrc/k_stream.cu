// k_stream.cu -- the weight-streaming expert kernels: every distinct routed expert and the
// shared expert stream their weights from HBM exactly once per call.
//
// Work: the gate/up launch (PHASE 0) runs, for each group of 32 intermediate columns j,
// the 32 gate + 32 up weight rows of the shared expert (bf16) and of every distinct routed
// expert d (MXFP4) against every row that uses them.  The down launch (PHASE 1) runs, for
// each group of 64 hidden outputs, the 64 w2 rows of the shared expert and of every
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
// Machine mapping (sm_103a):
//   * one CTA per SM, one producer warp + 8 consumer warps, items taken from a global
//     atomic counter (shared-expert items first, they are the largest);
//   * every pipeline stage holds one 64-row x 128-byte weight tile (256 MXFP4 or 64 bf16
//     elements per row), written by one or two 2D TMA loads with the 128-byte swizzle --
//     few, large TMA operations, since each one occupies the SM's TMA unit for a while;
//     the users' activation slices come with 1D bulk copies (routed) or one 2D box of all
//     rows (shared); the E8M0 and activation scales come with cp.async, all arriving on the
//     stage's mbarrier (transaction bytes + arrivals); 10 stages in flight per SM;
//   * consumer warp w works on MMA tile m = w & 3 (16 weight rows) and half h = w >> 2 of
//     every stage's K range: MXFP4 bytes go through cvt.rn.f16x2.e2m1x2 straight into
//     mma.m16n8k16 A fragments (weights = M rows, users = N columns), each 32-element
//     block's product is scaled by its E8M0 scale (times the activation block scale for
//     down) and accumulated in fp32; the shared expert is bf16 x bf16 into fp32;
//   * at the end of an item, tile m = (half 0) + (half 1), stored by one warp;
//   * activations enter the routed contractions as f16 with power-of-two scales (one per row
//     for gate/up, applied in the epilogue; one per 32-element block for down, applied per
//     block), exact for bf16 values in range;
//   * every mbarrier wait is bounded by a %globaltimer budget; on expiry the kernel sets
//     the status word and leaves.
#include "moe_tail_internal.cuh"

namespace mtail {

constexpr int kConsumerWarps = 8;
constexpr int kStreamThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 10;
constexpr int kChunkF4 = 256;            // MXFP4 elements per stage row (128 bytes)
constexpr int kChunkBF = 64;             // bf16 elements per stage row (128 bytes)
constexpr int kStageW = 8192;            // 64 weight rows x 128 bytes
constexpr int kActStride = 576;          // routed: bytes per user (512 + 64 pad)
constexpr int kStageA = kMaxRows * kActStride;
constexpr int kStageWS = 512;            // weight scales: 64 rows x 8 blocks
constexpr int kStageAS = kMaxRows * 32;  // activation scales: 16 users x 8 floats
constexpr int kStageBytes = kStageW + kStageA + kStageWS + kStageAS;
constexpr int kRedBytes = 2 * kConsumerWarps * 2 * 512;  // 2 x [warp][nt][lane] float4
constexpr int kTableBytes = (3 * kMaxPicks + 1 + kMaxRows) * 4;
constexpr int kXmaxBytes = 2 * 4 * kMaxRows * 4;
constexpr int kStreamSmem = kStages * kStageBytes + kRedBytes + 256 + kTableBytes + kXmaxBytes;

static_assert(kStageBytes % 1024 == 0, "stages stay 1024-byte aligned");

enum : int { kSharedGU = 0, kRoutedGU = 1, kSharedDN = 2, kRoutedDN = 3 };

struct Item {
  int kind;
  int e, d;
  int row0, row1;  // tensor-map rows: gate (or single) box, up box
  int out0;        // first output index (j for gate/up, h for down)
  int K, nst, chunk;
  int U, u0;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// The call's dedup tables, copied to shared memory once per CTA.
struct Tables {
  const int* uniq;      // [D] distinct expert ids
  const int* off;       // [D + 1] user offsets
  const int* users;     // [R*k] pick indices r*k + slot
  const float* rscale;  // [R] per-row scale of the f16 gate/up activations
};

__device__ __forceinline__ Item decode_item(int phase, int item, const Dims& dm,
                                            const Tables& s, int D) {
  Item it;
  it.d = 0;
  it.e = 0;
  it.u0 = 0;
  it.row1 = 0;
  if (phase == 0) {
    const int ns = dm.Is / 32;
    it.K = dm.H;
    if (item < ns) {
      it.kind = kSharedGU;
      it.out0 = item * 32;
      it.row0 = it.out0;
      it.row1 = dm.Is + it.out0;
      it.U = dm.R;
      it.chunk = kChunkBF;
    } else {
      const int q = item - ns, per = dm.I / 32;
      it.kind = kRoutedGU;
      it.d = min(q / per, D - 1);
      it.e = s.uniq[it.d];
      it.out0 = (q % per) * 32;
      it.row0 = it.e * 2 * dm.I + it.out0;
      it.row1 = it.row0 + dm.I;
      it.u0 = s.off[it.d];
      it.U = s.off[it.d + 1] - it.u0;
      it.chunk = kChunkF4;
    }
  } else {
    const int ns = dm.H / 64;
    if (item < ns) {
      it.kind = kSharedDN;
      it.K = dm.Is;
      it.out0 = item * 64;
      it.row0 = it.out0;
      it.U = dm.R;
      it.chunk = kChunkBF;
    } else {
      const int q = item - ns, per = dm.H / 64;
      it.kind = kRoutedDN;
      it.K = dm.I;
      it.d = min(q / per, D - 1);
      it.e = s.uniq[it.d];
      it.out0 = (q % per) * 64;
      it.row0 = it.e * dm.H + it.out0;
      it.u0 = s.off[it.d];
      it.U = s.off[it.d + 1] - it.u0;
      it.chunk = kChunkF4;
    }
  }
  it.U = max(0, min(it.U, kMaxRows));
  it.nst = (it.K + it.chunk - 1) / it.chunk;
  return it;
}

// ------------------------------------------------------------------ PTX wrappers ----

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)),
               "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* b) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(b))
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait: false when the budget ran out (the caller records the timeout).
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, uint64_t budget_ns) {
  if (mbar_try_wait(b, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(b, parity)) return true;
    if ((i & 63) == 0 && globaltimer() - t0 > budget_ns) return false;
  }
}
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ void lds128(uint32_t addr, uint32_t& a, uint32_t& b, uint32_t& c,
                                       uint32_t& d) {
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
               : "r"(addr));
}
__device__ __forceinline__ void mma_f16(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void cvt_e2m1x4(uint32_t w, uint32_t* h) {
  e2m1x8_to_f16x2(w, h[0], h[1], h[2], h[3]);
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Byte address of 16-byte chunk c of row r in a box of 64-byte rows written by TMA with
// the 64-byte swizzle (chunk index XOR bits 1..2 of the row; box base 512-byte aligned).
__device__ __forceinline__ uint32_t swz64(uint32_t base, int r, int c) {
  return base + (uint32_t)(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
}

// Byte offset of 16-byte chunk c of row r in a box of 128-byte rows written by TMA with the
// 128-byte swizzle (chunk index XOR the row's low 3 bits; box base 1024-byte aligned).
__device__ __forceinline__ int swz128_off(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

// d = A * B for one m16n8k16 f16 product (no accumulator input).
__device__ __forceinline__ void mma_f16_z(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// E8M0 byte i of a little-endian word of four scales -> float 2^(s-127); the byte 0
// (2^-127) flushes to 0.
__device__ __forceinline__ float e8m0_byte(uint32_t w, int i) {
  return __uint_as_float((i < 3 ? (w << (23 - 8 * i)) : (w >> 1)) & 0x7F800000u);
}

// Per-lane shared-memory offsets (within a stage), fixed for the kernel: warp cw works on
// MMA tile m = cw & 3 and on half h = cw >> 2 of every stage's K range.
struct Lane {
  // routed (MXFP4): word t of block chunk 4h + c, A rows g and g + 8; the 4 E8M0 bytes of
  // those rows for blocks 4h..4h+3; user g's 16 bytes of block 4h; down: user 2t's scales
  int code_a[4], code_b[4];
  int scale_a, scale_b;
  int act, ascale;
  // shared (bf16): chunk 2t + h of A rows g and g + 8; user g's matching 16 bytes
  int bw_a, bw_b, bact;
};

__device__ __forceinline__ Lane make_lane(bool gate_up, int cw, int g, int t) {
  Lane L;
  const int m = cw & 3, h = cw >> 2;
  int ra, rb, boxa, boxb, sra, srb;
  if (gate_up) {  // gate box rows 8m+g (A rows 0-7), up box rows 8m+g (A rows 8-15)
    ra = 8 * m + g; rb = ra;
    boxa = 0; boxb = 4096;
    sra = ra; srb = 32 + rb;
  } else {        // one 64-row box: rows 16m+g and 16m+g+8
    ra = 16 * m + g; rb = ra + 8;
    boxa = 0; boxb = 0;
    sra = ra; srb = rb;
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    L.code_a[c] = boxa + swz128_off(ra, 4 * h + c) + 4 * t;
    L.code_b[c] = boxb + swz128_off(rb, 4 * h + c) + 4 * t;
  }
  L.scale_a = kStageW + kStageA + sra * 8 + 4 * h;
  L.scale_b = kStageW + kStageA + srb * 8 + 4 * h;
  L.act = kStageW + g * kActStride + (4 * h) * 64 + t * 16;
  L.ascale = kStageW + kStageA + kStageWS + (2 * t) * 32 + 16 * h;
  L.bw_a = boxa + swz128_off(ra, 2 * t + h);
  L.bw_b = boxb + swz128_off(rb, 2 * t + h);
  L.bact = kStageW + swz128_off(g, 2 * t + h);
  return L;
}

// One stage of a routed MXFP4 item: 4 scale blocks x 1 tile per warp.  Each block's two
// k16 products are scaled by the row's E8M0 scale (and, for down, the user's block scale)
// and added to the fp32 accumulators.
template <bool GATE_UP>
__device__ __forceinline__ void stage_routed(const uint8_t* st, const Lane& L, int NT,
                                             float (&acc)[2][4]) {
  const uint32_t swa = *reinterpret_cast<const uint32_t*>(st + L.scale_a);
  const uint32_t swb = *reinterpret_cast<const uint32_t*>(st + L.scale_b);
  float4 as0[2], as1[2];  // down: scales of users (2t, 2t+1) for the 4 blocks, per N-tile
  if (!GATE_UP) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      if (nt < NT) {
        as0[nt] = *reinterpret_cast<const float4*>(st + L.ascale + nt * 8 * 32);
        as1[nt] = *reinterpret_cast<const float4*>(st + L.ascale + nt * 8 * 32 + 32);
      }
    }
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t wa = *reinterpret_cast<const uint32_t*>(st + L.code_a[c]);
    const uint32_t wb = *reinterpret_cast<const uint32_t*>(st + L.code_b[c]);
    uint32_t ha[4], hb[4];
    e2m1x8_to_f16x2(wa, ha[0], ha[1], ha[2], ha[3]);
    e2m1x8_to_f16x2(wb, hb[0], hb[1], hb[2], hb[3]);
    const float sa = e8m0_byte(swa, c), sb = e8m0_byte(swb, c);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      if (nt < NT) {
        const uint4 b = *reinterpret_cast<const uint4*>(st + L.act + nt * 8 * kActStride + c * 64);
        float tmp[4];
        mma_f16_z(tmp, ha[0], hb[0], ha[1], hb[1], b.x, b.y);
        mma_f16(tmp, ha[2], hb[2], ha[3], hb[3], b.z, b.w);
        if (GATE_UP) {
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
}

// One stage of a shared-expert (bf16) item: 32 K elements (half h) x 1 tile per warp.
// Lane t takes elements [16t + 8h, +8) of the 64-element stage row, for its two A rows and
// for user g (conflict-free under the 128-byte swizzle).
__device__ __forceinline__ void stage_shared(const uint8_t* st, const Lane& L, int NT,
                                             float (&acc)[2][4]) {
  const uint4 a = *reinterpret_cast<const uint4*>(st + L.bw_a);
  const uint4 c = *reinterpret_cast<const uint4*>(st + L.bw_b);
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    if (nt < NT) {
      // users 8..15 are rows 8..15 of the activation box: same swizzle phase as rows 0..7
      const uint4 b = *reinterpret_cast<const uint4*>(st + L.bact + nt * 8 * 128);
      mma_bf16(acc[nt], a.x, c.x, a.y, c.y, b.x, b.y);
      mma_bf16(acc[nt], a.z, c.z, a.w, c.w, b.z, b.w);
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
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) set_status(s.status, kStatusBadTile);
    return;
  }
  uint8_t* stages = smem;
  float4* red = (float4*)(smem + kStages * kStageBytes);
  uint64_t* full = (uint64_t*)(smem + kStages * kStageBytes + kRedBytes);
  uint64_t* empty = full + kStages;
  int* info = (int*)(empty + kStages);  // [kStages][2]: item, k-chunk
  int* t_uniq = (int*)(smem + kStages * kStageBytes + kRedBytes + 256);
  int* t_off = t_uniq + kMaxPicks;
  int* t_users = t_off + kMaxPicks + 1;
  float* t_rscale = (float*)(t_users + kMaxPicks);
  float* xmax = t_rscale + kMaxRows;  // [2][4 tiles][kMaxRows]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Before the routing is known: pull this CTA's share of the shared expert's weights into
  // L2 (they do not depend on any earlier kernel), so their HBM reads overlap the front.
  if (warp == 0) {
    const uint8_t* base = (PHASE == 0) ? (const uint8_t*)w.ws13 : (const uint8_t*)w.ws2;
    const size_t total = (size_t)dm.Is * dm.H * 2 * (PHASE == 0 ? 2 : 1);
    const size_t per = ((total / gridDim.x) + 4095) & ~(size_t)4095;
    const size_t beg = (size_t)blockIdx.x * per;
    const size_t end = min(total, beg + per);
    for (size_t o = beg + (size_t)lane * 16384; o < end; o += 32 * 16384) {
      const uint32_t n = (uint32_t)min((size_t)16384, end - o);
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(base + o), "r"(n) : "memory");
    }
  }
  pdl_wait();
  const int D = min(max(*s.n_distinct, 1), kMaxPicks);
  const int n_items = (PHASE == 0) ? dm.Is / 32 + D * (dm.I / 32) : dm.H / 64 + D * (dm.H / 64);
  for (int i = threadIdx.x; i < D; i += kStreamThreads) t_uniq[i] = s.uniq[i];
  for (int i = threadIdx.x; i <= D; i += kStreamThreads) t_off[i] = s.user_off[i];
  for (int i = threadIdx.x; i < dm.R * dm.k; i += kStreamThreads) t_users[i] = s.user_list[i];
  for (int i = threadIdx.x; i < dm.R; i += kStreamThreads) t_rscale[i] = s.n16s[i];
  Tables tb;
  tb.uniq = t_uniq;
  tb.off = t_off;
  tb.users = t_users;
  tb.rscale = t_rscale;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1 + 32);
      mbar_init(&empty[i], kConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();

  if (warp == 0) {
    // ---------------------------------------------------------------- producer ----
    const uint64_t pol = policy_evict_first();
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    // stages whose copies were issued and not yet seen consumed, with their phase parity
    uint32_t pend = 0u, pend_par = 0u;
    // failure-injection switch: CTA 0 leaves its first stage unpublished, so the consumers'
    // bounded wait on it expires (tests the timeout path; never set in production)
    bool skip_first = (debug & kDebugStallFirstStage) && blockIdx.x == 0;
    int item = 0;
    if (lane == 0) item = (int)atomicAdd(&s.counters[PHASE], 1u);
    for (;;) {
      item = __shfl_sync(0xffffffffu, item, 0);
      if (item >= n_items) {
        pdl_trigger();  // this CTA is in its tail: let the next launch take the SM
        break;
      }
      int next = 0;  // the following item, fetched while this one streams
      if (lane == 0) next = (int)atomicAdd(&s.counters[PHASE], 1u);
      const Item it = decode_item(PHASE, item, dm, tb, D);
      const bool routed = (it.kind == kRoutedGU || it.kind == kRoutedDN);
      // lane u < U of a routed item: where user u's activations (and down's per-block
      // scales) come from
      const uint8_t* asrc = nullptr;
      const float* ssrc = nullptr;
      if (routed && lane < it.U) {
        if (it.kind == kRoutedGU) {
          asrc = (const uint8_t*)(s.n16 + (size_t)(tb.users[it.u0 + lane] / dm.k) * dm.H);
        } else {
          const int pick = tb.users[it.u0 + lane];
          asrc = (const uint8_t*)(s.mid16 + (size_t)pick * dm.I);
          ssrc = s.mid16s + (size_t)pick * (dm.I / 32);
        }
      }
      const uint8_t* wsbase = (it.kind == kRoutedGU) ? w.w13s : w.w2s;
      const int kb = it.K / 32;  // scale bytes per weight row
      for (int kc = 0; kc < it.nst && ok; ++kc) {
        if (lane == 0) ok = mbar_wait(&empty[stage], phase ^ 1, budget_ns);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        pend &= ~(1u << stage);
        if (skip_first) {
          skip_first = false;
          if (++stage == kStages) { stage = 0; phase ^= 1; }
          continue;
        }
        pend |= 1u << stage;
        pend_par = (pend_par & ~(1u << stage)) | (phase << stage);
        uint8_t* st = stages + stage * kStageBytes;
        uint8_t* sw = st;
        uint8_t* sa = st + kStageW;
        uint8_t* sws = sa + kStageA;
        uint8_t* sas = sws + kStageWS;
        const int k0 = kc * it.chunk;
        const int kval = min(it.chunk, it.K - k0);  // routed: 128 or 256; shared: 64
        if (lane == 0) {
          info[stage * 2] = item;
          info[stage * 2 + 1] = kc;
          uint32_t bytes = kStageW;  // full boxes, also when partly past K (zero filled)
          if (routed) bytes += (uint32_t)it.U * (uint32_t)kval * 2u;
          else bytes += (uint32_t)dm.Rmax * 128u;
          mbar_expect_tx(&full[stage], bytes);
          if (it.kind == kRoutedGU) {
            tma_load_2d(sw, &maps.w13, k0 >> 1, it.row0, &full[stage], pol);
            tma_load_2d(sw + 4096, &maps.w13, k0 >> 1, it.row1, &full[stage], pol);
          } else if (it.kind == kRoutedDN) {
            tma_load_2d(sw, &maps.w2, k0 >> 1, it.row0, &full[stage], pol);
          } else if (it.kind == kSharedGU) {
            tma_load_2d(sw, &maps.ws13, k0, it.row0, &full[stage], pol);
            tma_load_2d(sw + 4096, &maps.ws13, k0, it.row1, &full[stage], pol);
            tma_load_2d(sa, &maps.n, k0, 0, &full[stage], 0ull);
          } else {
            tma_load_2d(sw, &maps.ws2, k0, it.row0, &full[stage], pol);
            tma_load_2d(sa, &maps.ms, k0, 0, &full[stage], 0ull);
          }
        }
        __syncwarp();
        if (routed) {
          // user u's f16 activation slice, by lane u
          if (lane < it.U)
            bulk_load(sa + lane * kActStride, asrc + (size_t)k0 * 2, (uint32_t)kval * 2u,
                      &full[stage]);
          // E8M0 scales of the 64 weight rows, 8 blocks each (4 bytes per copy)
          const int words = kval / 128;  // 1 or 2 words per row in this stage
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int c = lane + 32 * q;
            const int row = c >> 1, wd = c & 1;
            if (wd < words) {
              const size_t grow = (it.kind == kRoutedGU)
                                      ? ((row < 32) ? (size_t)it.row0 + row : (size_t)it.row1 + (row - 32))
                                      : (size_t)it.row0 + row;
              cp_async4(sws + row * 8 + wd * 4, wsbase + grow * kb + (k0 / 32) + wd * 4);
            }
          }
          // per-block activation scales (down only: the gate/up activations carry one
          // scale per row, applied in the epilogue)
          if (ssrc != nullptr) {
            for (int half = 0; half < words; ++half)
              cp_async16(sas + lane * 32 + half * 16, ssrc + k0 / 32 + half * 4);
          }
        }
        cp_async_arrive_noinc(&full[stage]);
        if (++stage == kStages) { stage = 0; phase ^= 1; }
      }
      if (!ok) break;
      item = next;
    }
    if (ok) {
      // end-of-work marker
      if (lane == 0) ok = mbar_wait(&empty[stage], phase ^ 1, budget_ns);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (ok) {
        if (lane == 0) {
          info[stage * 2] = -1;
          info[stage * 2 + 1] = 0;
          mbar_arrive(&full[stage]);
        }
        cp_async_arrive_noinc(&full[stage]);
      }
    }
    if (!ok) {
      // a wait expired: record it, then let every copy this CTA issued land (bounded)
      // before the CTA's shared memory is released
      if (lane == 0) {
        set_status(s.status, kStatusTimeout);
        for (int st2 = 0; st2 < kStages; ++st2)
          if (pend & (1u << st2)) mbar_wait(&full[st2], (pend_par >> st2) & 1u, budget_ns);
      }
      __syncwarp();
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    return;
  }

  // ------------------------------------------------------------------ consumers ----
  const int cw = warp - 1;
  const int g = lane >> 2, t = lane & 3;
  const int em = cw & 3, eh = cw >> 2;  // this warp's tile and K half
  int stage = 0;
  uint32_t phase = 0;
  int cur = -1, nitems = 0;
  Item it;
  it.kind = 0; it.nst = 0; it.U = 0; it.K = 0; it.out0 = 0; it.u0 = 0; it.row0 = 0; it.row1 = 0;
  it.e = 0; it.d = 0; it.chunk = kChunkF4;
  const Lane L = make_lane(PHASE == 0, cw, g, t);
  float acc[2][4];
  for (;;) {
    if (!mbar_wait(&full[stage], phase, budget_ns)) {
      if (lane == 0) set_status(s.status, kStatusTimeout);
      break;
    }
    const int item = info[stage * 2], kc = info[stage * 2 + 1];
    if (item < 0) break;
    if (item != cur) {
      cur = item;
      it = decode_item(PHASE, item, dm, tb, D);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[nt][q] = 0.f;
    }
    const uint8_t* st = stages + stage * kStageBytes;
    const int NT = it.U > 8 ? 2 : 1;
    // this warp's half of the stage's K range starts at element (chunk / 2) * eh
    if (kc * it.chunk + (it.chunk >> 1) * eh < it.K) {
      if (it.kind == kRoutedGU || it.kind == kRoutedDN) {
        if (PHASE == 0) stage_routed<true>(st, L, NT, acc);
        else stage_routed<false>(st, L, NT, acc);
      } else {
        stage_shared(st, L, NT, acc);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
    if (++stage == kStages) { stage = 0; phase ^= 1; }

    if (kc == it.nst - 1) {
      // ------------------------------------------------------ item epilogue ----
      // partial sums go to one of two reduction buffers (alternating by item, so the next
      // item's writes need no barrier); tile m = (half 0) + (half 1), i.e. warps m and
      // m + 4, finished by warp m + 4 * nt for N-tile nt.
      const int buf = nitems & 1;
      ++nitems;
      float4* rb = red + buf * (kConsumerWarps * 2 * 32);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
        if (nt < NT)
          rb[(cw * 2 + nt) * 32 + lane] = make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
      named_bar_sync(1, kConsumerWarps * 32);
      const int ent = eh;  // N-tile this warp finishes
      const bool active = ent < NT;
      float c[4] = {0.f, 0.f, 0.f, 0.f};
      if (active) {
        const float4 v0 = rb[(em * 2 + ent) * 32 + lane];
        const float4 v1 = rb[((em + 4) * 2 + ent) * 32 + lane];
        c[0] = v0.x + v1.x; c[1] = v0.y + v1.y; c[2] = v0.z + v1.z; c[3] = v0.w + v1.w;
      }
      if (it.kind == kSharedGU) {
        if (active) {
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int r = ent * 8 + 2 * t + q;
            if (r < it.U)
              s.ms[(size_t)r * dm.Is + it.out0 + 8 * em + g] =
                  __float2bfloat16_rn(silu_f(c[q]) * c[2 + q]);
          }
        }
      } else if (it.kind == kSharedDN) {
        if (active) {
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int r = ent * 8 + 2 * t + q;
            if (r < it.U) {
              float* yrow = s.ys + (size_t)r * dm.H + it.out0 + 16 * em;
              yrow[g] = c[q];
              yrow[g + 8] = c[2 + q];
            }
          }
        }
      } else if (it.kind == kRoutedDN) {
        if (active) {
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int u = ent * 8 + 2 * t + q;
            if (u < it.U) {
              float* yrow = s.y + (size_t)tb.users[it.u0 + u] * dm.H + it.out0 + 16 * em;
              yrow[g] = c[q];
              yrow[g + 8] = c[2 + q];
            }
          }
        }
      } else {
        // routed gate/up: mid = bf16(SiLU(gate) * up) with the row's activation scale
        // restored; its f16 copy gets one power-of-two scale per (pick, 32 columns), from
        // the maximum over the item's 4 tiles (exchanged through shared memory)
        float* mx = xmax + buf * (4 * kMaxRows);
        float mv[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int u = ent * 8 + 2 * t + q;
          const float rs = (active && u < it.U) ? tb.rscale[tb.users[it.u0 + u] / dm.k] : 0.f;
          mv[q] = __bfloat162float(__float2bfloat16_rn(silu_f(c[q] * rs) * (c[2 + q] * rs)));
          float amax = fabsf(mv[q]);
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 8));
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 16));
          if (active && g == 0) mx[em * kMaxRows + u] = amax;
        }
        named_bar_sync(2, kConsumerWarps * 32);
        if (active) {
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int u = ent * 8 + 2 * t + q;
            if (u < it.U) {
              float amax = 0.f;
#pragma unroll
              for (int m2 = 0; m2 < 4; ++m2) amax = fmaxf(amax, mx[m2 * kMaxRows + u]);
              int p = 0;
              if (amax > 0.f) {
                const int ex = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127;
                p = max(-100, min(100, ex - 14));
              }
              const float down = __uint_as_float((uint32_t)(127 - p) << 23);
              const int pick = tb.users[it.u0 + u];
              s.mid16[(size_t)pick * dm.I + it.out0 + 8 * em + g] = __float2half_rn(mv[q] * down);
              if (em == 0 && g == 0)
                s.mid16s[(size_t)pick * (dm.I / 32) + it.out0 / 32] =
                    __uint_as_float((uint32_t)(127 + p) << 23);
            }
          }
        }
      }
    }
  }
}

// Opt the streaming kernels in to their shared-memory size (once per process and device
// before the first launch; called at create time, outside any graph capture).
cudaError_t prepare_stream_kernels() {
  cudaError_t e = cudaFuncSetAttribute(k_stream<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kStreamSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_stream<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kStreamSmem);
  return e;
}

cudaError_t launch_stream(int phase, const StreamMaps& maps, const Dims& d, const Weights& w,
                          const Scratch& s, int num_sms, uint64_t budget_ns, cudaStream_t st,
                          bool pdl, uint32_t debug) {
  if (phase == 0)
    return launch_k(k_stream<0>, dim3(num_sms), dim3(kStreamThreads), kStreamSmem, st, pdl,
                    maps, d, w, s, budget_ns, debug);
  return launch_k(k_stream<1>, dim3(num_sms), dim3(kStreamThreads), kStreamSmem, st, pdl, maps,
                  d, w, s, budget_ns, debug);
}

// ----------------------------------------------------------- tensor-map encoding ----

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static int encode_2d(EncodeTiledFn fn, CUtensorMap* m, CUtensorMapDataType dt, const void* base,
                     uint64_t inner, uint64_t rows, uint64_t row_bytes, uint32_t box_inner,
                     uint32_t box_rows) {
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : -1;
}

// Every box has 128-byte rows (the 128-byte swizzle span): 128 MXFP4 code bytes (256
// elements) or 64 bf16 elements.  Returns 0 on success, -1 if the driver has no tensor-map
// encoder, -2 if encoding failed.
int make_stream_maps(StreamMaps* out, const Dims& d, const Weights& w, const Scratch& s) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess || fn == nullptr)
    return -1;
  EncodeTiledFn enc = (EncodeTiledFn)fn;
  const uint64_t H = d.H, E = d.E, I = d.I, Is = d.Is, R = d.Rmax;
  const CUtensorMapDataType U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8, BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  if (encode_2d(enc, &out->w13, U8, w.w13c, H / 2, E * 2 * I, H / 2, 128, 32)) return -2;
  if (encode_2d(enc, &out->w2, U8, w.w2c, I / 2, E * H, I / 2, 128, 64)) return -2;
  if (encode_2d(enc, &out->ws13, BF, w.ws13, H, 2 * Is, H * 2, 64, 32)) return -2;
  if (encode_2d(enc, &out->ws2, BF, w.ws2, Is, H, Is * 2, 64, 64)) return -2;
  if (encode_2d(enc, &out->n, BF, s.n, H, R, H * 2, 64, (uint32_t)R)) return -2;
  if (encode_2d(enc, &out->ms, BF, s.ms, Is, R, Is * 2, 64, (uint32_t)R)) return -2;
  return 0;
}

}  // namespace mtail
