// k_stream_tc.cu -- the weight-streaming expert kernels on the fifth-generation tensor cores:
// each routed MXFP4 expert runs as tcgen05 block-scaled MMAs (kind::mxf4: E2M1 x E2M1 with
// one E8M0 scale per 32 elements on both operands), the bf16 shared expert as tcgen05
// kind::f16 MMAs; accumulators live in tensor memory.
//
// Work items, their order and the launch synchronisation are those of the CUDA-core form
// (k_stream.cu): gate/up items of 64 gate + 64 up weight rows, down items of 128 weight
// rows, each distinct routed expert streamed once per call, shared-expert items first;
// down items wait (bounded) for the gate/up items of their expert, the combine for the down
// items of its 128 outputs.
//
// Sources: "[AMD] integrate kimi k3 monokernel" page, Kernel Replacement rows "The routed
// experts" and "The shared expert gate_up / SiLU and mul / down"; "glm53: Long-context
// indexer ..." page, Modifications rows 16 (every using row a column of one multi-column
// product per expert), 17, 18 and 21.
//
// Swap-AB: the weights are the MMA's A operand (M = 128 rows, K-major, exactly the
// 128-byte-swizzled TMA boxes of the CUDA-core form); the activations are B (N columns).
// The tensor core's block-scaled MXFP4 product needs E2M1 on both sides, so every bf16
// activation row enters as four E2M1 planes with their own per-32 E8M0 scales: plane 0 is
// the nearest E2M1 multiple of a power of two sized to the block maximum, each further plane
// the same for what the planes before it left over.  Each plane gains about two bits; four
// leave a remainder below ~1e-3 of the block maximum (the output error is far smaller, the
// remainders being independent).  A row of activations is thus four B columns (plane-major
// within the row), and the epilogue adds the four column sums in plane order.  The norm
// launch writes the planes of n; the gate/up epilogue writes the planes of mid.
//
// Scales: the MMAs read E8M0 scales from tensor memory, brought there by tcgen05.cp from
// scale-factor atoms in shared memory (512 bytes: 4 blocks of 128 rows, see sf_atom_offset).
// Every scale a stage needs arrives as such atoms with the stage: the weights' from a copy of
// w13s / w2s laid out in atoms once at create (1 KB of contiguous bytes per stage and weight
// tile), the activation planes' as written in atoms by the launch that makes them (the norm for
// n, the gate/up epilogue for mid, per distinct expert).  So no thread rearranges scales on the
// way, and the scale bytes stream as whole kilobytes instead of 64-byte pieces of 128 rows.
//
// Machine mapping (sm_103a), one CTA of 224 threads per SM.  A tcgen05.mma or tcgen05.cp
// costs its issuing thread a fixed ~75 ns whatever N is (measured on GB300), while the
// tensor core keeps up with several issuers at once; so two threads issue, each owning half
// of every stage's K and an accumulator of its own, and nothing else runs on them:
//   * warp 0, lane 0 -- the producer: per stage one TMA load of a 128-row x 128-byte weight
//     tile (L2 evict-first), one TMA load of the activation tile (planes, or bf16 rows for the
//     shared expert), and for a routed item the stage's weight and activation scale atoms
//     (two bulk copies of 1 KB);
//   * warps 1, 2 (lane 0) -- the MMA issuers: issuer h copies scale-factor atom h of the
//     stage's weights and activations into its own tensor-memory columns (tcgen05.cp) and
//     issues the two MMAs of K steps 2h, 2h + 1 (K = 64 FP4 or 16 bf16 elements each; 32
//     bytes of every operand row) into its accumulator, then commits the stage;
//   * warps 3..6 -- the epilogue: tcgen05.ld of both accumulators (TMEM lane = weight row)
//     added in issuer order, plane sums, SiLU * up through a shared-memory exchange between
//     the gate and up lane quadrants, planes of mid, stores, and the counts the next launch
//     waits for;
//   * tensor memory (512 columns): two accumulator slots x two issuers x N columns, and a
//     ring of per-stage scale-factor slots (16 columns each); every wait is bounded, and a
//     CTA that gives up lets its copies and MMAs finish before it frees its tensor memory.
#include <algorithm>
#include <cstring>

#include "k_combine.cuh"
#include "k_front.cuh"
#include "k_persist.cuh"
#include "k_stream_common.cuh"

namespace mtail {

// warps: producer, two MMA issuers, four epilogue warps (warp mod 4 = their lane quadrant)
constexpr int kTcWarpMma = 1, kTcWarpEpi = 3;
constexpr int kTcThreads = 7 * 32;
constexpr int kTcSfBytes = 2048;    // per stage: A atoms 2 x 512 B, B atoms 2 x 512 B
constexpr int kTcCols = 512;        // tensor-memory columns of a CTA
constexpr int kTcSfCol = 256;       // first scale-factor column (accumulators below)
constexpr int kTcMaxStages = 12;    // 16 scale-factor columns each: 256 + 192 <= 512
constexpr uint32_t kNamedBarEpi = 1;
// bf16 (shared-expert) MMA columns: the call's rows, 16 up to 16 rows, 32 above
template <int NMAX>
constexpr int kSharedCols = NMAX <= 64 ? 16 : 32;
// accumulator slots: two (an item's MMAs overlap the previous item's epilogue), one at 128
// columns (two issuers x 128 columns fill the half of tensor memory the slots may use)
template <int NMAX>
constexpr int kAccSlots = NMAX <= 64 ? 2 : 1;

// --------------------------------------------------------------------- PTX wrappers ----

__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo,
                                              uint32_t layout) {
  // tcgen05 shared-memory matrix descriptor: start, leading and stride byte offsets (>> 4),
  // descriptor version 1, layout type in bits 61..63 (2 = 128-byte swizzle, 0 = none)
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)layout << 61);
}
// K-major operand rows of 128 bytes under the 128-byte swizzle (8-row atoms 1024 bytes apart)
__device__ __forceinline__ uint64_t sw128_desc(const void* p) {
  return smem_desc(smem_u32(p), 16, 1024, 2);
}
// scale-factor atom: 32 rows x 16 bytes, contiguous (no swizzle; 8-row groups 128 bytes apart)
__device__ __forceinline__ uint64_t sf_desc(const void* p) { return smem_desc(smem_u32(p), 128, 128, 0); }

// Instruction descriptors.  kind::mxf4: E2M1 operands (format 1), K-major, N >> 3 at bit 17,
// UE8M0 scales (bit 23), M >> 4 at bit 24; the scale-factor byte of A at bits 29..30 and of B
// at bits 4..5.  kind::f16: fp32 accumulator (bit 4), bf16 operands (format 1).
__device__ __forceinline__ uint32_t idesc_mxf4(int N, uint32_t sf_id) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) | (8u << 24) |
         (sf_id << 29) | (sf_id << 4);
}
__device__ __forceinline__ uint32_t idesc_bf16(int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | (8u << 24);
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc));
}
__device__ __forceinline__ void tc_mma_mxf4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                            uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], "
      "[%6], p;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb));
}
__device__ __forceinline__ void tc_mma_f16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                           uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
// arrive on `bar` once every tcgen05 operation this thread issued so far has completed
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void mbar_arrive_n(uint64_t* b, uint32_t n) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(n)
               : "memory");
}
__device__ __forceinline__ void bar_epi() {
  asm volatile("bar.sync %0, %1;" ::"n"(kNamedBarEpi), "n"(128) : "memory");
}

// 32 lanes x 16/32/64 consecutive fp32 columns of the accumulator (lane = TMEM lane).
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float (&v)[N]);

#define MT_R4(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3])
template <>
__device__ __forceinline__ void tmem_ld<16>(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : MT_R4(0), MT_R4(4), MT_R4(8), MT_R4(12)
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
template <>
__device__ __forceinline__ void tmem_ld<32>(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : MT_R4(0), MT_R4(4), MT_R4(8), MT_R4(12), MT_R4(16), MT_R4(20), MT_R4(24), MT_R4(28)
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
template <>
__device__ __forceinline__ void tmem_ld<64>(uint32_t taddr, float (&v)[64]) {
  float a[32], b[32];
  tmem_ld<32>(taddr, a);
  tmem_ld<32>(taddr + 32, b);
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    v[i] = a[i];
    v[32 + i] = b[i];
  }
}
#undef MT_R4

// ----------------------------------------------------------- E2M1 activation planes ----
// (the norm launch makes the planes of n with the same two helpers, see k_front.cu)

// --------------------------------------------------------------- shared-memory plan ----

struct TcPtrs {
  uint8_t* stages;   // [stages][16 KB weights, b_bytes activations, 2 KB scale atoms]
  float* xch;        // [2][2][64][Rmax]: gate and up sums of a gate/up item, two buffers
  int* t_uniq;
  int* t_off;
  int* t_users;
  uint64_t* full;    // [stages] producer -> MMA issuers (transaction bytes)
  uint64_t* empty;   // [stages] MMA commits (2) -> producer
  uint64_t* afull;   // [2] MMA commits (2) + item id (1) -> epilogue: accumulators ready
  uint64_t* aempty;  // [2] epilogue (4 warps) -> MMA issuers: accumulators read
  uint64_t* drain;   // [2] an issuer's own commit, only when its CTA gives up
  int2* info;        // [stages] item of each stage
  int* aitem;        // [2] item of each accumulator slot
  uint32_t* tbase;   // tensor-memory base address of the CTA
  int* eflag;        // epilogue: this CTA completed a split shared item
  int* sD;           // the call's distinct-expert count once the tables are in shared memory
  uint64_t* tables;  // [1] epilogue warps -> producer: routing tables copied (gate/up launch)
};

// set: which of the two barrier sets (the persistent launch's down roles take the second, so
// that no arrival still landing on a barrier of its gate/up roles meets a new one)
__device__ __forceinline__ TcPtrs tc_carve(uint8_t* smem, const TcLayout& L, int set) {
  TcPtrs p;
  p.stages = smem;
  p.xch = reinterpret_cast<float*>(smem + L.off_x);
  p.t_uniq = reinterpret_cast<int*>(smem + L.off_tab);
  p.t_off = p.t_uniq + L.tab_picks;
  p.t_users = p.t_off + L.tab_picks + 1;
  p.full = reinterpret_cast<uint64_t*>(smem + L.off_bar + set * L.bar_set_bytes);
  p.empty = p.full + kTcMaxStages;
  p.afull = p.empty + kTcMaxStages;
  p.aempty = p.afull + 2;
  p.drain = p.aempty + 2;
  p.tables = p.drain + 2;
  p.info = reinterpret_cast<int2*>(p.tables + 1);
  p.aitem = reinterpret_cast<int*>(p.info + kTcMaxStages);
  p.tbase = reinterpret_cast<uint32_t*>(p.aitem + 2);
  p.eflag = reinterpret_cast<int*>(p.tbase + 1);
  p.sD = p.eflag + 1;
  return p;
}

// K parts of every shared-expert gate/up item of this call: the fewest (1, 2 or 4, dividing
// H / 64) that bring an item down to an SM's share of the launch's bytes (so that at one or a
// few rows the shared items do not outlast the routed ones) and give three quarters of the
// CTAs a shared part to stream until the routing is known (a CTA whose first item is routed
// waits for the router's tables).  Computed on the host at launch (64-bit divisions).
static int shared_parts(const Dims& dm, int D, int nsm) {
  const int ns = dm.Is / 64;
  if (ns > kMaxSharedSplitItems) return 1;
  const uint64_t item_b = 128ull * (uint64_t)dm.H * 2;
  const uint64_t routed_b = 128ull * (uint64_t)(dm.H / 2 + dm.H / 32);
  const uint64_t total = (uint64_t)ns * item_b + (uint64_t)D * (uint64_t)(dm.I / 64) * routed_b;
  const uint64_t share = total / (uint64_t)nsm;
  int p = 1;
  while (p < kMaxSharedParts && (dm.H / 64) % (2 * p) == 0 &&
         (item_b / (uint64_t)p > share || 4 * ns * p < 3 * nsm))
    p *= 2;
  return p;
}

// Items of a launch when the shared gate/up items are split into P K parts: the ns * P parts
// first (part = item mod P, K elements [part H / P, (part + 1) H / P)), then the routed items.
__device__ __forceinline__ Item decode_tc(int phase, int item, const Dims& dm, const Tables& tb,
                                          int D, int P) {
  if (phase != 0 || P == 1) return decode_item(phase, item, dm, tb, D);
  const int ns = dm.Is / 64;
  if (item < ns * P) {
    Item it = decode_item(0, item / P, dm, tb, D);
    it.part = item % P;
    it.K = dm.H / P;
    it.k0 = it.part * it.K;
    it.nst = it.K / kChunkBF;
    return it;
  }
  return decode_item(0, item - ns * (P - 1), dm, tb, D);
}

// ----------------------------------------------------------------------- epilogue ----

// Sum of the four plane columns of activation column group c (plane order).
template <int N>
__device__ __forceinline__ float plane_sum(const float (&v)[N], int c) {
  return ((v[4 * c] + v[4 * c + 1]) + v[4 * c + 2]) + v[4 * c + 3];
}

// The four E2M1 planes of one 32-element block of mid held one element per lane (lane =
// element), stored as plane rows of the down launch's activations: 16 code bytes at
// `codes + p * code_pitch` and one scale byte at `scales + p * scale_pitch`.
__device__ __forceinline__ void store_planes_lane(float v, int lane, uint8_t* codes,
                                                  size_t code_pitch, uint8_t* scales,
                                                  size_t scale_pitch) {
  float r = v;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    float am = fabsf(r);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    const int e = e2m1_plane_exp(am);
    const uint32_t code = e2m1_code(r * exp2_int(-e));
    r -= e2m1_value(code) * exp2_int(e);
    // eight codes per 32-bit word, element 2j in the low nibble of byte j
    uint32_t w = code << (4 * (lane & 7));
    w |= __shfl_xor_sync(0xffffffffu, w, 1);
    w |= __shfl_xor_sync(0xffffffffu, w, 2);
    w |= __shfl_xor_sync(0xffffffffu, w, 4);
    if ((lane & 7) == 0)
      *reinterpret_cast<uint32_t*>(codes + p * code_pitch + (lane >> 1)) = w;
    if (lane == 0) scales[p * scale_pitch] = (uint8_t)(e + 127);
  }
}

// One finished item: its accumulator (N plane columns per TMEM lane) to outputs.
// C columns (16 or 32) of an item's sums from column c0: issuer 0's accumulator plus issuer
// 1's, in that order, when issuer 1 took part (it owns the second 128 K elements of every
// stage).  Loading 32 columns at most at a time bounds the registers at 128 columns.
template <int C>
__device__ __forceinline__ void acc_chunk(uint32_t acc0, uint32_t acc1, bool two, int c0,
                                          float (&v)[C]) {
  tmem_ld<C>(acc0 + (uint32_t)c0, v);
  if (two) {
    float w[C];
    tmem_ld<C>(acc1 + (uint32_t)c0, w);
#pragma unroll
    for (int i = 0; i < C; ++i) v[i] += w[i];
  }
}

template <int NMAX>
__device__ __forceinline__ bool tc_finish(const Item& it, int item, int P, uint32_t acc0,
                                          uint32_t acc1, float* xch, int* eflag, int ew, int q,
                                          int lane, const Dims& dm, const Tables& tb,
                                          const Scratch& s) {
  // bf16 items have whole 64-element stages; an MXFP4 item's first stage reaches past 128
  // elements unless K is 128
  const bool two = (it.kind == kSharedGU || it.kind == kSharedDN) || it.K > 128;
  const int m = 32 * q + lane;  // weight row of this thread within the item's 128
  constexpr int NSH = kSharedCols<NMAX>;  // bf16 (shared-expert) columns: the rows
  if (it.kind == kRoutedGU || it.kind == kSharedGU) {
    const int R = dm.Rmax;
    // [R][64] gate sums, then [R][64] up sums: a warp's 32 lanes (weight rows) store, and the
    // SiLU tasks' lanes (outputs) load, 32 consecutive words
    float* xg = xch;
    float* xu = xch + 64 * R;
    float* dst = (m < 64) ? xg + m : xu + (m - 64);
    if (it.kind == kSharedGU && P > 1) {
      // one K part: its sums to scratch; the CTA whose part completes the item adds all parts
      // in part order (whichever CTAs ran them) and finishes it
      const int si = item / P;
      float v[NSH];
      acc_chunk<NSH>(acc0, acc1, true, 0, v);
      float* gp = s.gpart + ((size_t)(si * kMaxSharedParts + it.part) * 128 + m) * R;
#pragma unroll
      for (int c = 0; c < NSH; ++c)
        if (c < R) gp[c] = v[c];
      __threadfence();
      bar_epi();
      if (ew == 0 && lane == 0)
        *eflag = (atomicAdd(&s.counters[kCtrSharedParts + si], 1u) == (uint32_t)(P - 1)) ? 1 : 0;
      bar_epi();
      if (!*eflag) return false;
      __threadfence();
      const float* g0 = s.gpart + ((size_t)(si * kMaxSharedParts) * 128 + m) * R;
#pragma unroll
      for (int c = 0; c < NSH; ++c) {
        if (c < R) {
          float a = __ldcg(g0 + c);
          for (int pp = 1; pp < P; ++pp) a += __ldcg(g0 + (size_t)pp * 128 * R + c);
          dst[c * 64] = a;
        }
      }
    } else if (it.kind == kRoutedGU) {
      // columns 4r + p: row r's planes, 32 columns (8 rows) at a time
      constexpr int C = NMAX < 32 ? NMAX : 32;
#pragma unroll
      for (int c0 = 0; c0 < NMAX; c0 += C) {
        if (c0 / 4 < R) {
          float v[C];
          acc_chunk<C>(acc0, acc1, two, c0, v);
#pragma unroll
          for (int c = 0; c < C / 4; ++c)
            if (c0 / 4 + c < R) dst[(c0 / 4 + c) * 64] = plane_sum<C>(v, c);
        }
      }
    } else {
      float v[NSH];
      acc_chunk<NSH>(acc0, acc1, two, 0, v);
#pragma unroll
      for (int c = 0; c < NSH; ++c)
        if (c < R) dst[c * 64] = v[c];
    }
    bar_epi();
    if (it.kind == kRoutedGU) {
      // (user, 32-column block) tasks, one per warp at a time; lane = column in the block
      for (int t = ew; t < 2 * it.U; t += 4) {
        const int u = t >> 1, blk = t & 1;
        const int slot = it.u0 + u;
        const int r = tb.users[slot] / dm.k;
        const int j = 32 * blk + lane;
        const float g = xg[r * 64 + j], up = xu[r * 64 + j];
        const float mv = __bfloat162float(__float2bfloat16_rn(silu_f(g) * up));
        const size_t cp = (size_t)dm.I / 2;
        // scales: atoms of this expert's down items, column 4 u + p (the planes of a user
        // stay inside one 32-column group, so plane p is 16 bytes after plane 0)
        uint8_t* sa = s.mid4a + (size_t)it.d * sf_atoms_per_tile(dm.I) * 512 +
                      sf_atom_offset(4 * u, (it.out0 + 32 * blk) / 32);
        store_planes_lane(mv, lane, s.mid4 + (size_t)(4 * slot) * cp + (it.out0 + 32 * blk) / 2,
                          cp, sa, 16);
      }
    } else {
      for (int e = 32 * ew + lane; e < 64 * dm.R; e += 128) {
        const int j = e & 63, r = e >> 6;
        s.ms[(size_t)r * dm.Is + it.out0 + j] =
            __float2bfloat16_rn(silu_f(xg[r * 64 + j]) * xu[r * 64 + j]);
      }
    }
  } else if (it.kind == kRoutedDN) {
    // columns 4u + p: user u's planes, 32 columns (8 users) at a time
    constexpr int C = NMAX < 32 ? NMAX : 32;
#pragma unroll
    for (int c0 = 0; c0 < NMAX; c0 += C) {
      if (c0 / 4 < it.U) {
        float v[C];
        acc_chunk<C>(acc0, acc1, two, c0, v);
#pragma unroll
        for (int c = 0; c < C / 4; ++c) {
          const int u = c0 / 4 + c;
          if (u < it.U) s.y[(size_t)tb.users[it.u0 + u] * dm.H + it.out0 + m] = plane_sum<C>(v, c);
        }
      }
    }
  } else {  // shared down
    float v[NSH];
    acc_chunk<NSH>(acc0, acc1, two, 0, v);
#pragma unroll
    for (int r = 0; r < NSH; ++r)
      if (r < dm.R) s.ys[(size_t)r * dm.H + it.out0 + m] = v[r];
  }
  return true;
}

// ------------------------------------------------------------------------ kernel ----

// The persistent launch's arguments (zero in the multi-kernel launches).
struct PersistArgs {
  const __nv_bfloat16* x;
  __nv_bfloat16* residual;
  __nv_bfloat16* out;
  RouterPlan rp;
  int stall;  // failure injection: CTA 0 leaves at once, the others' barrier waits expire
  uint32_t* done;  // host-visible completion word (signal_done), or null
  uint32_t seq;
  const HostArgs* ha;  // a host-buffer call: x, residual, out and seq from here instead
};

// The expert roles of one CTA over the items of launch phases PH0..PH1 (0 = gate/up, 1 =
// down): one phase per launch in the multi-kernel form (PH0 == PH1); in the single persistent
// launch (PH0 = 0, PH1 = 1) the gate/up roles and then, shared and tensor memory set up afresh
// with a second barrier set, the down roles, between the front and the combine below.
// --------------------------------------------------------- single persistent launch ----
// The whole call in one cooperative launch of one CTA per SM (224 threads, the streaming
// kernels' shared-memory plan): add + RMSNorm (CTA r takes row r), a grid barrier, the
// router's parts as virtual CTAs spread over the grid (the last part ranks the experts,
// builds the dedup tables and publishes them), then the expert roles of the streaming
// kernels over the gate/up items and, once none is left, over the down items (a CTA starts on
// its shared-expert items at once; routed items wait for the published routing, down items
// for the gate/up items of their expert), then the combine (each warp waits for the down items
// of its outputs).  Only the norm -> router hand-over is a grid barrier; every later one is
// a count per expert or per output tile, as between the launches of the multi-kernel form.
// Sources: "[AMD] integrate kimi k3 monokernel" page, Motivation and Kernel Replacement (the
// layer tail as one resident launch whose stages hand over through in-kernel flags); "Split
// the Kimi3 AttnRes mix across CTAs for decode rows" page (a tag per call instead of a
// reset, here the barrier's generation word).
template <int PH0, int PH1, int NMAX, bool FRONT>
__global__ void __launch_bounds__(kTcThreads, 1)
k_stream_tc(const __grid_constant__ TcMaps maps, Dims dm, Weights w, Scratch s,
            uint64_t budget_ns, uint32_t debug, PersistArgs pa) {
  extern __shared__ __align__(1024) uint8_t smem[];
  constexpr bool kPersist = FRONT;  // the single persistent launch: front, experts, combine
  constexpr bool kBoth = PH0 != PH1;  // gate/up roles, then down roles, in the same CTA
  // failure-injection switch of the persistent launch (never set in production)
  if (kPersist && pa.stall && blockIdx.x == 0) return;
  // the tensor maps this CTA's copies will use (all encoded at create; mid4[i] for boxes of
  // at most NMAX rows), fetched while the rest of the set-up runs
  if (threadIdx.x < 32) {
    const CUtensorMap* m = nullptr;
    const int l = threadIdx.x;
    if (PH0 == 0 && l < 4) m = l == 0 ? &maps.w13 : l == 1 ? &maps.np4 : l == 2 ? &maps.ws13 : &maps.n;
    if (PH1 == 1 && l >= 4 && l < 8 && (16 << (l - 4)) <= NMAX) m = &maps.mid4[l - 4];
    if (PH1 == 1 && l >= 8 && l < 11) m = l == 8 ? &maps.w2 : l == 9 ? &maps.ws2 : &maps.ms;
    if (m) asm volatile("prefetch.tensormap [%0];" ::"l"(m) : "memory");
  }
  // the persistent launch's buffers (a host-buffer call's from its arguments)
  const __nv_bfloat16* px = pa.x;
  __nv_bfloat16* pres = pa.residual;
  __nv_bfloat16* pout = pa.out;
  uint32_t pseq = pa.seq;
  if (kPersist && pa.ha) {  // read once per CTA (host memory: every access crosses the link)
    __shared__ const void* s_buf[3];
    __shared__ uint32_t s_seq;
    if (threadIdx.x == 0) {
      s_buf[0] = ha_ptr(&pa.ha->x);
      s_buf[1] = ha_ptr((const void* const*)&pa.ha->residual);
      s_buf[2] = ha_ptr((const void* const*)&pa.ha->out);
      s_seq = *reinterpret_cast<const volatile uint32_t*>(&pa.ha->seq);
    }
    __syncthreads();
    px = reinterpret_cast<const __nv_bfloat16*>(s_buf[0]);
    pres = reinterpret_cast<__nv_bfloat16*>(const_cast<void*>(s_buf[1]));
    pout = reinterpret_cast<__nv_bfloat16*>(const_cast<void*>(s_buf[2]));
    pseq = s_seq;
  }
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) set_status(s.status, kStatusBadTile);
    return;  // (persistent launch: the other CTAs' barrier waits expire)
  }
  if constexpr (kPersist) {
    __shared__ float part[kTcThreads / 32];
    __shared__ int s_last;
    if (threadIdx.x == 0) tl_first(s.tl, kTlNormStart);
    // 1. the call's counter words (not the barrier's); this CTA's first router part's weights
    //    (they depend on nothing); add + RMSNorm, each row split over P CTAs.  The residual is
    //    read here and rewritten by the combine, after the barrier below.
    if (blockIdx.x == 0)
      for (int i = threadIdx.x; i < kCtrWords; i += kTcThreads)
        if (i != kCtrPersistArrive && i != kCtrPersistGen) s.counters[i] = 0u;
    const int nparts = pa.rp.tiles * pa.rp.parts;
    if ((int)blockIdx.x < nparts)
      router_stage_w<kTcThreads>(smem, w.w_r, blockIdx.x % pa.rp.tiles, blockIdx.x / pa.rp.tiles,
                                 pa.rp.plen, dm.H, dm.E);
    // (a host-buffer call reads x and residual over the host link: at most 4 CTAs per row
    // read each row, so that the whole-row reads for rstd stay small there)
    const int P = max(1, min(min((int)gridDim.x / dm.R, dm.H / 256), pa.ha ? 4 : kMaxNormParts));
    for (int v = blockIdx.x; v < dm.R * P; v += gridDim.x)
      add_rmsnorm_part<kTcThreads>(v % dm.R, v / dm.R, P, px, pres, w.gamma, s.rnew,
                                   s.n, dm.H, dm.eps, w.wsg,
                                   s.gate_part + (size_t)(v % dm.R) * kMaxNormParts, s.np4,
                                   s.np4a, part);
    if (threadIdx.x == 0 && (int)blockIdx.x < dm.R * P) tl_last(s.tl, kTlNormEnd);
    if (!grid_barrier(s, budget_ns)) return;
    // each row's gate from its parts' logits, added in part order (before this CTA's router
    // ticket, which orders it before every later reader)
    if (w.wsg && blockIdx.x == 0)
      for (int r = threadIdx.x; r < dm.R; r += kTcThreads) {
        float z = 0.f;
        for (int q = 0; q < P; ++q) z += __ldcg(s.gate_part + (size_t)r * kMaxNormParts + q);
        s.sgate[r] = 1.0f / (1.0f + expf(-z));
      }
    // 2. the router's parts (the first one's weights are already on their way)
    if (threadIdx.x == 0) {
      tl_first(s.tl, kTlRouterStart);
      if ((int)blockIdx.x < nparts) tl_last(s.tl, kTlRouterAllStarted);
    }
    for (int v = blockIdx.x; v < nparts; v += gridDim.x) {
      const int tile = v % pa.rp.tiles, p = v / pa.rp.tiles;
      if (v != (int)blockIdx.x)
        router_stage_w<kTcThreads>(smem, w.w_r, tile, p, pa.rp.plen, dm.H, dm.E);
      if (router_part<kTcThreads / 32>(smem, s, tile, p, pa.rp.plen, pa.rp.red_off, dm.R, dm.H,
                                       dm.E, (uint32_t)nparts, &s_last))
        router_finish<kTcThreads, true>(smem, s, pa.rp.parts, dm.R, dm.E, dm.k);
      __syncthreads();
    }
    // The expert roles' copies read activations written with ordinary stores earlier in this
    // launch (n and its planes, before the barrier; the producer is thread 0, which took the
    // barrier's acquire): order those writes first.
    if (threadIdx.x == 0) {
      asm volatile("fence.proxy.async.global;" ::: "memory");
      tl_first(s.tl, kTlGateUpStart);
    }
  } else {
    if (threadIdx.x == 0) tl_first(s.tl, PH0 == 0 ? kTlGateUpStart : kTlDownStart);
  }
#pragma unroll
  for (int PHASE = PH0; PHASE <= PH1; ++PHASE) {
  if (kBoth && PHASE == 1 && threadIdx.x == 0) tl_first(s.tl, kTlDownStart);
  // trigger: release the next launch once the barriers are set up (multi-kernel form);
  // bar_set: the persistent launch's down roles take the second barrier set, so that no
  // arrival still landing on a barrier of its gate/up roles meets a new one; last: the CTA
  // allocates no tensor memory after this phase (it gives up its allocation permit)
  const bool trigger = !kPersist;
  const int bar_set = (kBoth && PHASE == 1) ? 1 : 0;
  const bool last = PHASE == PH1;
  const TcLayout& lay = maps.lay;
  const TcPtrs sp = tc_carve(smem, lay, bar_set);
  const int S = lay.stages;
  constexpr uint32_t A = kAccSlots<NMAX>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Gate/up items start while the router still runs (the shared-expert items need only n,
  // complete before the router's wait returned): the shared items are split by the call's
  // largest possible distinct count, and the routed items wait for the tables (copied to
  // shared memory by the epilogue warps once the router's last CTA has published them).  A
  // down-only launch starts after every gate/up CTA, and waits for the published routing once
  // before it reads the tables.
  const int P = (PHASE == 0) ? dm.sparts : 1;
  const int n_shared = (PHASE == 0) ? (dm.Is / 64) * P : 0;  // items that need no routing
  int D = 1, n_items = 0;
  if (PHASE == 1) {
    if (threadIdx.x == 0 && !wait_count(&s.counters[kCtrRouted], 1u, budget_ns))
      set_status(s.status, kStatusTimeout);
    __syncthreads();
    D = min(max(__ldcg(s.n_distinct), 1), kMaxPicks);
    for (int i = threadIdx.x; i < D; i += kTcThreads) sp.t_uniq[i] = __ldcg(s.uniq + i);
    for (int i = threadIdx.x; i <= D; i += kTcThreads) sp.t_off[i] = __ldcg(s.user_off + i);
    for (int i = threadIdx.x; i < dm.R * dm.k; i += kTcThreads)
      sp.t_users[i] = __ldcg(s.user_list + i);
    if (threadIdx.x == 0) *sp.sD = D;
    n_items = items_of(1, dm, D);
  }
  Tables tb;
  tb.uniq = sp.t_uniq;
  tb.off = sp.t_off;
  tb.users = sp.t_users;
  tb.rscale = nullptr;

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&sp.full[i], 1);
      mbar_init(&sp.empty[i], 2);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sp.afull[i], 3);
      mbar_init(&sp.aempty[i], 4);
      mbar_init(&sp.drain[i], 1);
    }
    mbar_init(sp.tables, 1);
    if (PHASE == 0) *sp.sD = 1;  // until the routing is known (only routed items read it)
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (trigger) pdl_trigger();  // the next launch may queue for SMs (it waits on counts)
  }
  if (warp == kTcWarpMma) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(sp.tbase)),
                 "n"(kTcCols));
    if (last) asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *sp.tbase;
  bool ok = true;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer ----
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t pend = 0u, pend_par = 0u;
      bool skip_first = PHASE == 0 && (debug & kDebugStallFirstStage) && blockIdx.x == 0;
      bool stamped = false, stamped_routed = false;  // timeline stamps taken (tracing only)
      // scale atoms per weight tile: over H (gate/up) or I (down), two per stage
      const int ga = sf_atoms_per_tile(PHASE == 0 ? dm.H : dm.I);
      // a CTA's first item is its index, later ones come from the counter (from gridDim.x on);
      // the persistent launch's gate/up items all come from the counter (its CTAs reach those
      // roles at different times: the ones without a router part first)
      const bool claim_all = kPersist && PHASE == 0;
      const int base = claim_all ? 0 : (int)gridDim.x;
      int item = claim_all ? (int)atomicAdd(&s.counters[work_counter(PHASE)], 1u) : (int)blockIdx.x;
      bool have_tables = (PHASE == 1);
      bool gu_all = false;  // every gate/up item of the call counted (down roles)
      while (ok) {
        if (!have_tables && item >= n_shared) {
          // the first routed item: the routing tables must be in shared memory
          if (!mbar_wait(sp.tables, 0, budget_ns)) { ok = false; break; }
          have_tables = true;
          D = *sp.sD;
          n_items = n_shared + D * (dm.I / 64);
        }
        if (have_tables && item >= n_items) break;
        const int next = base + (int)atomicAdd(&s.counters[work_counter(PHASE)], 1u);
        const Item it = decode_tc(PHASE, item, dm, tb, D, P);
        const bool routed = (it.kind == kRoutedGU || it.kind == kRoutedDN);
        const int hsel = (it.U <= 4) ? 0 : (it.U <= 8) ? 1 : (it.U <= 16) ? 2 : 3;
        const int nb = (it.kind == kRoutedGU) ? NMAX : (it.kind == kRoutedDN) ? (16 << hsel) : 0;
        if (PHASE == 1 && !gu_all) {
          // the item's inputs (the shared expert's or its expert's mid): wait for their gate/up
          // items, then order the async proxy's reads after them; once every gate/up item of
          // the call is counted, one such fence covers all later items.  Both counts are read
          // together (relaxed), the fence after them takes the acquire side of their releases.
          const bool sh = (it.kind == kSharedDN);
          const uint32_t* cd = &s.counters[sh ? kCtrSharedGUDone : kCtrGUDone + it.d];
          const uint32_t need = (uint32_t)(sh ? dm.Is / 64 : dm.I / 64);
          uint32_t va, vd;
          asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(va)
                       : "l"(&s.counters[kCtrGUAllDone]) : "memory");
          asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(vd) : "l"(cd) : "memory");
          if (va >= (uint32_t)(D * (dm.I / 64) + dm.Is / 64)) {
            gu_all = true;
          } else if (vd < need && !wait_count(cd, need, budget_ns)) {
            ok = false;
            break;
          }
          asm volatile("fence.acq_rel.gpu;" ::: "memory");
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        // the item's scale atoms: its weight tile's (expert e, tile t) and its activations'
        const uint8_t* a_sf = nullptr;
        const uint8_t* b_sf = nullptr;
        if (it.kind == kRoutedGU) {
          const int e = it.row0 / (2 * dm.I), t = it.out0 / 64;
          a_sf = w.w13a + (size_t)(e * (dm.I / 64) + t) * ga * 512;
          b_sf = s.np4a;
        } else if (it.kind == kRoutedDN) {
          const int e = it.row0 / dm.H, t = it.out0 / 128;
          a_sf = w.w2a + (size_t)(e * (dm.H / 128) + t) * ga * 512;
          b_sf = s.mid4a + (size_t)it.d * ga * 512;
        }
        const uint32_t b_bytes = routed ? (uint32_t)nb * 128u : (uint32_t)dm.Rmax * 128u;
        const uint32_t bytes = kStageW + b_bytes + (routed ? (uint32_t)kTcSfBytes : 0u);
        for (int kc = 0; kc < it.nst; ++kc) {
          if (!mbar_wait(&sp.empty[stage], phase ^ 1, budget_ns)) { ok = false; break; }
          pend &= ~(1u << stage);
          if (skip_first) {
            skip_first = false;
            if (++stage == S) { stage = 0; phase ^= 1; }
            continue;
          }
          uint8_t* st = sp.stages + stage * lay.stage_bytes;
          uint8_t* sb = st + kStageW;
          uint8_t* sa = sb + lay.b_bytes;
          pend |= 1u << stage;
          pend_par = (pend_par & ~(1u << stage)) | (phase << stage);
          sp.info[stage] = make_int2(item, 0);
          mbar_expect_tx(&sp.full[stage], bytes);
          if (s.tl) {  // each CTA's first copy, and its first of a routed gate/up item
            if (!stamped) {
              tl_first(s.tl, PHASE == 0 ? kTlGateUpFirstCopy : kTlDownFirstCopy);
              if (PHASE == 0) tl_last(s.tl, kTlGateUpAllCopying);
            }
            if (!stamped_routed && PHASE == 0 && it.kind == kRoutedGU) {
              tl_first(s.tl, kTlGateUpRouted);
              stamped_routed = true;
            }
            stamped = true;
          }
          if (it.kind == kRoutedGU) {
            // the 64 gate and 64 up rows in one copy (3-D box over [2E][I][H/2])
            const int x = kc * (kChunkF4 / 2);
            tma_load_3d(st, &maps.w13, x, it.out0, 2 * (it.row0 / (2 * dm.I)), &sp.full[stage],
                        pol);
            tma_load_2d(sb, &maps.np4, x, 0, &sp.full[stage]);
          } else if (it.kind == kRoutedDN) {
            const int x = kc * (kChunkF4 / 2);
            tma_load_2d(st, &maps.w2, x, it.row0, &sp.full[stage], pol);
            tma_load_2d(sb, &maps.mid4[hsel], x, 4 * it.u0, &sp.full[stage]);
          } else if (it.kind == kSharedGU) {
            const int x = it.k0 + kc * kChunkBF;
            tma_load_3d(st, &maps.ws13, x, it.out0, 0, &sp.full[stage], pol);
            tma_load_2d(sb, &maps.n, x, 0, &sp.full[stage]);
          } else {
            tma_load_2d(st, &maps.ws2, kc * kChunkBF, it.row0, &sp.full[stage], pol);
            tma_load_2d(sb, &maps.ms, kc * kChunkBF, 0, &sp.full[stage]);
          }
          if (routed) {
            // atoms 2 kc and 2 kc + 1 of the weights (A), then of the activations (B)
            bulk_load(sa, a_sf + (size_t)kc * 1024, 1024u, &sp.full[stage], pol);
            bulk_load(sa + 1024, b_sf + (size_t)kc * 1024, 1024u, &sp.full[stage]);
          }
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
        item = next;
      }
      if (ok) {
        ok = mbar_wait(&sp.empty[stage], phase ^ 1, budget_ns);
        if (ok && !skip_first) {
          sp.info[stage] = make_int2(-1, 0);
          mbar_arrive(&sp.full[stage]);
        }
      }
      if (!ok) {
        set_status(s.status, kStatusTimeout);
        for (int st2 = 0; st2 < S; ++st2)
          if (pend & (1u << st2)) mbar_wait(&sp.full[st2], (pend_par >> st2) & 1u, budget_ns);
      }
    }
  } else if (warp >= kTcWarpMma && warp < kTcWarpEpi) {
    // ------------------------------------------------------------ MMA issuers ----
    // issuer h owns K steps 2h and 2h + 1 of every stage (the second half of its 256 MXFP4
    // or 64 bf16 elements for h = 1): its scale atoms, its MMAs, its own accumulator
    const int h = warp - kTcWarpMma;
    int stage = 0;
    uint32_t phase = 0, acnt = 0;
    int kc = 0;
    Item it;
    it.nst = 0;
    for (;;) {
      if (!mbar_wait(&sp.full[stage], phase, budget_ns)) { ok = false; break; }
      const int item = sp.info[stage].x;
      if (item < 0) break;
      if (kc == 0) {
        it = decode_tc(PHASE, item, dm, tb, *sp.sD, P);
        if (!mbar_wait(&sp.aempty[acnt % A], ((acnt / A) & 1u) ^ 1u, budget_ns)) {
          ok = false;
          break;
        }
      }
      tc_fence_after();
      const bool routed = (it.kind == kRoutedGU || it.kind == kRoutedDN);
      if (lane == 0) {
        const uint8_t* st = sp.stages + stage * lay.stage_bytes;
        const uint8_t* sb = st + kStageW;
        const uint32_t acc = tbase + (2u * (acnt % A) + (uint32_t)h) * (uint32_t)NMAX;
        if (routed) {
          const int hsel = (it.U <= 4) ? 0 : (it.U <= 8) ? 1 : (it.U <= 16) ? 2 : 3;
          const int nb = (it.kind == kRoutedGU) ? NMAX : (16 << hsel);
          const uint8_t* atoms = sb + lay.b_bytes;
          const uint32_t sf = tbase + kTcSfCol + 16u * (uint32_t)stage + 8u * (uint32_t)h;
          tc_cp_sf(sf, sf_desc(atoms + 512 * h));          // A atom h: blocks 4h..4h+3
          tc_cp_sf(sf + 4, sf_desc(atoms + 1024 + 512 * h));  // B atom h
          const int nk = min(4, (it.K - kc * kChunkF4 + 63) / 64);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int kk = 2 * h + j;
            if (kk < nk)
              tc_mma_mxf4(acc, sw128_desc(st + 32 * kk), sw128_desc(sb + 32 * kk),
                          idesc_mxf4(nb, 2u * (uint32_t)j), sf, sf + 4,
                          (kc > 0 || j > 0) ? 1u : 0u);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int kk = 2 * h + j;
            tc_mma_f16(acc, sw128_desc(st + 32 * kk), sw128_desc(sb + 32 * kk),
                       idesc_bf16(kSharedCols<NMAX>),
                       (kc > 0 || j > 0) ? 1u : 0u);
          }
        }
        tc_commit(&sp.empty[stage]);
      }
      __syncwarp();
      if (++stage == S) { stage = 0; phase ^= 1; }
      if (++kc == it.nst) {
        // this issuer's accumulator is final once its MMAs complete; issuer 0 also
        // publishes the item id (three arrivals in all)
        if (lane == 0) {
          if (h == 0) sp.aitem[acnt % A] = item;
          tc_commit(&sp.afull[acnt % A]);
          if (h == 0) mbar_arrive(&sp.afull[acnt % A]);
        }
        __syncwarp();
        ++acnt;
        kc = 0;
      }
    }
    if (ok && h == 0) {
      // end of work: an end marker in the next accumulator slot
      if (mbar_wait(&sp.aempty[acnt % A], ((acnt / A) & 1u) ^ 1u, budget_ns)) {
        if (lane == 0) {
          sp.aitem[acnt % A] = -1;
          mbar_arrive_n(&sp.afull[acnt % A], 3);
        }
      } else {
        ok = false;
      }
    }
    if (!ok) {
      // let every MMA and copy this thread issued finish before the memory is released
      if (lane == 0) {
        set_status(s.status, kStatusTimeout);
        tc_commit(&sp.drain[h]);
        mbar_wait(&sp.drain[h], 0, budget_ns);
      }
      __syncwarp();
    }
  } else {
    // --------------------------------------------------------------- epilogue ----
    const int q = warp & 3, ew = warp - kTcWarpEpi;
    if (PHASE == 0) {
      // the routing: wait for the tables the router's last CTA publishes, copy them into
      // shared memory, and release the producer's routed items (none if the wait expired)
      if (ew == 0 && lane == 0) {
        int dv = 0;
        if (wait_count(&s.counters[kCtrRouted], 1u, budget_ns))
          dv = min(max(__ldcg(s.n_distinct), 1), kMaxPicks);
        else
          set_status(s.status, kStatusTimeout);
        *sp.eflag = dv;
      }
      bar_epi();
      const int dv = *sp.eflag;
      const int et = 32 * ew + lane;
      if (dv > 0) {
        for (int i = et; i < dv; i += 128) sp.t_uniq[i] = __ldcg(s.uniq + i);
        for (int i = et; i <= dv; i += 128) sp.t_off[i] = __ldcg(s.user_off + i);
        for (int i = et; i < dm.R * dm.k; i += 128) sp.t_users[i] = __ldcg(s.user_list + i);
      }
      bar_epi();
      if (et == 0) {
        *sp.sD = dv;
        mbar_arrive(sp.tables);
      }
    }
    for (uint32_t ac = 0;; ++ac) {
      const uint32_t as = ac % A;
      if (!mbar_wait(&sp.afull[as], (ac / A) & 1u, budget_ns)) {
        if (lane == 0) set_status(s.status, kStatusTimeout);
        break;
      }
      tc_fence_after();
      const int item = sp.aitem[as];
      if (item < 0) break;
      const Item it = decode_tc(PHASE, item, dm, tb, *sp.sD, P);
      const uint32_t lq = (uint32_t)(32 * q) << 16;
      const uint32_t acc0 = tbase + (2u * as) * (uint32_t)NMAX + lq;
      const uint32_t acc1 = tbase + (2u * as + 1u) * (uint32_t)NMAX + lq;
      float* xch = sp.xch;  // one buffer: the item-end barrier orders its reuse
      const bool done = tc_finish<NMAX>(it, item, P, acc0, acc1, xch, sp.eflag, ew, q, lane, dm,
                                        tb, s);
      // every epilogue thread's stores before the count the next launch waits for: the
      // epilogue barrier orders them before the counting thread's fence and release
      tc_fence_before();
      bar_epi();
      if (done && ew == 0 && lane == 0) {
        uint32_t* c = &s.counters[PHASE == 1 ? kCtrTileDone + it.out0 / 128
                                  : it.kind == kSharedGU ? kCtrSharedGUDone
                                                         : kCtrGUDone + it.d];
        __threadfence();
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(c) : "memory");
        if (PHASE == 0)
          asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(&s.counters[kCtrGUAllDone])
                       : "memory");
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sp.aempty[as]);
    }
  }

  // every role ends here: tensor memory is freed once all of them are done with it
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) tl_last(s.tl, PHASE == 0 ? kTlGateUpEnd : kTlDownEnd);
  if (warp == kTcWarpMma) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase),
                 "n"(kTcCols));
  }
  }
  if constexpr (kPersist) {
    // 4. the combine: thread t of the grid takes 8-output groups t, t + grid threads, ...
    if (threadIdx.x == 0) tl_first(s.tl, kTlCombineStart);
    const int ng = dm.H / 8;  // a multiple of 32: a warp's groups lie in one row
    for (int u = blockIdx.x * kTcThreads + threadIdx.x; u < dm.R * ng; u += gridDim.x * kTcThreads) {
      const int r = u / ng, c = u % ng;
      if (!combine_wait_tiles(s, c, budget_ns)) break;  // whole warps
      combine_one(dm, s, r, c, pout, pres, w.wsg != nullptr);
    }
    if ((threadIdx.x & 31) == 0) tl_last(s.tl, kTlCombineEnd);
    signal_done(s, pa.done, pseq, gridDim.x);
  }
}

template <int NMAX>
static cudaError_t persist_prepare_one(int* blocks, int* smem_limit) {
  cudaFuncAttributes a;
  cudaError_t e = cudaFuncGetAttributes(&a, k_stream_tc<0, 1, NMAX, true>);
  if (e != cudaSuccess) return e;
  *smem_limit = kSmemLimit - (int)a.sharedSizeBytes;
  e = cudaFuncSetAttribute(k_stream_tc<0, 1, NMAX, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           *smem_limit);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks, k_stream_tc<0, 1, NMAX, true>, kTcThreads,
                                                      *smem_limit);
  return e;
}

cudaError_t persistent_smem_limit(int nmax, int* smem_limit) {
  int blocks = 0;
  if (nmax == 16) return persist_prepare_one<16>(&blocks, smem_limit);
  if (nmax == 32) return persist_prepare_one<32>(&blocks, smem_limit);
  if (nmax == 64) return persist_prepare_one<64>(&blocks, smem_limit);
  return persist_prepare_one<128>(&blocks, smem_limit);
}

cudaError_t persistent_prepare(const TcMaps& maps, int* blocks_per_sm) {
  int limit = 0;
  const int nmax = maps.lay.nmax;
  if (nmax == 16) return persist_prepare_one<16>(blocks_per_sm, &limit);
  if (nmax == 32) return persist_prepare_one<32>(blocks_per_sm, &limit);
  if (nmax == 64) return persist_prepare_one<64>(blocks_per_sm, &limit);
  return persist_prepare_one<128>(blocks_per_sm, &limit);
}

template <int NMAX>
static cudaError_t persist_launch(const TcMaps& maps, const Dims& d, const __nv_bfloat16* x,
                                  __nv_bfloat16* residual, __nv_bfloat16* out, const Weights& w,
                                  const Scratch& s, int grid, const RouterPlan& rp, size_t smem,
                                  uint64_t budget_ns, int stall, cudaStream_t st, uint32_t* done,
                                  uint32_t seq, const HostArgs* ha) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  PersistArgs pa;
  pa.x = x;
  pa.residual = residual;
  pa.out = out;
  pa.rp = rp;
  pa.stall = stall;
  pa.done = done;
  pa.seq = seq;
  pa.ha = ha;
  return cudaLaunchKernelEx(&cfg, k_stream_tc<0, 1, NMAX, true>, maps, d, w, s, budget_ns, 0u, pa);
}

cudaError_t launch_persistent(const TcMaps& maps, const Dims& d, const __nv_bfloat16* x,
                              __nv_bfloat16* residual, __nv_bfloat16* out, const Weights& w,
                              const Scratch& s, int grid, uint64_t budget_ns, bool stall,
                              cudaStream_t st, uint32_t* done, uint32_t seq,
                              const HostArgs* ha) {
  const RouterPlan rp = router_plan(d.R, d.H, d.E, kTcThreads / 32);
  // the front's use of the same shared memory: gamma (2 H bytes), a router part, the last
  // part's logits and top-k workspace
  const size_t topk = (((size_t)d.R * d.E * 4 + 15) & ~(size_t)15) + kTopkWsBytes;
  const size_t smem = std::max(std::max((size_t)maps.lay.smem_bytes, rp.smem),
                               std::max((size_t)d.H * 2, topk));
  const int nmax = maps.lay.nmax, st_ = stall ? 1 : 0;
  Dims dd = d;
  dd.sparts = shared_parts(d, std::min(d.E, d.R * d.k), grid);
  if (nmax == 16) return persist_launch<16>(maps, dd, x, residual, out, w, s, grid, rp, smem, budget_ns, st_, st, done, seq, ha);
  if (nmax == 32) return persist_launch<32>(maps, dd, x, residual, out, w, s, grid, rp, smem, budget_ns, st_, st, done, seq, ha);
  if (nmax == 64) return persist_launch<64>(maps, dd, x, residual, out, w, s, grid, rp, smem, budget_ns, st_, st, done, seq, ha);
  return persist_launch<128>(maps, dd, x, residual, out, w, s, grid, rp, smem, budget_ns, st_, st, done, seq, ha);
}

cudaError_t persistent_reset(const Scratch& s) {
  return cudaMemset(s.counters + kCtrPersistArrive, 0, 2 * sizeof(uint32_t));
}

// -------------------------------------------------------------------- host side ----

template <int PH0, int PH1, int NMAX>
static cudaError_t tc_prepare_one() {
  return cudaFuncSetAttribute(k_stream_tc<PH0, PH1, NMAX, false>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
}

template <int PH0, int PH1>
static cudaError_t tc_prepare_phases() {
  cudaError_t e = tc_prepare_one<PH0, PH1, 16>();
  if (e == cudaSuccess) e = tc_prepare_one<PH0, PH1, 32>();
  if (e == cudaSuccess) e = tc_prepare_one<PH0, PH1, 64>();
  if (e == cudaSuccess) e = tc_prepare_one<PH0, PH1, 128>();
  return e;
}

cudaError_t prepare_stream_tc_kernels() {
  cudaError_t e = tc_prepare_phases<0, 0>();
  if (e == cudaSuccess) e = tc_prepare_phases<1, 1>();
  return e;
}

template <int PH0, int PH1, int NMAX>
static cudaError_t tc_launch(const TcMaps& maps, const Dims& d, const Weights& w,
                             const Scratch& s, int num_sms, uint64_t budget_ns, cudaStream_t st,
                             bool pdl, uint32_t debug) {
  return launch_k(k_stream_tc<PH0, PH1, NMAX, false>, dim3(num_sms), dim3(kTcThreads),
                  (size_t)maps.lay.smem_bytes, st, pdl, maps, d, w, s, budget_ns, debug,
                  PersistArgs{});
}

template <int PH0, int PH1>
static cudaError_t tc_launch_n(const TcMaps& maps, const Dims& d, const Weights& w,
                               const Scratch& s, int num_sms, uint64_t budget_ns, cudaStream_t st,
                               bool pdl, uint32_t debug) {
  const int nmax = maps.lay.nmax;
  if (nmax == 16) return tc_launch<PH0, PH1, 16>(maps, d, w, s, num_sms, budget_ns, st, pdl, debug);
  if (nmax == 32) return tc_launch<PH0, PH1, 32>(maps, d, w, s, num_sms, budget_ns, st, pdl, debug);
  if (nmax == 64) return tc_launch<PH0, PH1, 64>(maps, d, w, s, num_sms, budget_ns, st, pdl, debug);
  return tc_launch<PH0, PH1, 128>(maps, d, w, s, num_sms, budget_ns, st, pdl, debug);
}

// phase 0: gate/up, 1: down.  (One launch of both phases, a CTA taking down items once no
// gate/up item is left, measured slower at every row count: 0.8 us at 8 rows, 4.4 at 1, 3.6
// at 16, 9.3 at 32.)
cudaError_t launch_stream_tc(int phase, const TcMaps& maps, const Dims& d, const Weights& w,
                             const Scratch& s, int num_sms, uint64_t budget_ns, cudaStream_t st,
                             bool pdl, uint32_t debug) {
  if (phase == 0) {
    Dims dd = d;
    dd.sparts = shared_parts(d, std::min(d.E, d.R * d.k), num_sms);
    return tc_launch_n<0, 0>(maps, dd, w, s, num_sms, budget_ns, st, pdl, debug);
  }
  return tc_launch_n<1, 1>(maps, d, w, s, num_sms, budget_ns, st, pdl, debug);
}

// Shared-memory plan: stages of 16 KB weights + nmax x 128 B activations + 2 KB scale atoms,
// as many as fit (up to kTcMaxStages, the tensor-memory scale ring), the epilogue exchange,
// the dedup tables and the barriers.
TcLayout make_tc_layout(int Rmax, int k, int smem_limit) {
  TcLayout L;
  L.nmax = (Rmax <= 4) ? 16 : (Rmax <= 8) ? 32 : (Rmax <= 16) ? 64 : 128;
  L.aslots = (L.nmax <= 64) ? 2 : 1;
  L.tab_picks = Rmax * k;
  L.b_bytes = L.nmax * 128;
  L.stage_bytes = kStageW + L.b_bytes + kTcSfBytes;
  const int x_bytes = 2 * 64 * Rmax * 4;
  const int tab_bytes = ((3 * L.tab_picks + 1) * 4 + 127) & ~127;
  // mbarriers full, empty per stage + afull, aempty, drain (2 each) + tables; the stages'
  // item words; the accumulator slots' item words; tbase, eflag and sD
  // (two sets of them)
  const int bar_bytes = (2 * kTcMaxStages + 7) * 8 + kTcMaxStages * 8 + 2 * 4 + 4 + 4 + 4;
  L.bar_set_bytes = (bar_bytes + 127) & ~127;
  const int fixed = x_bytes + tab_bytes + 2 * L.bar_set_bytes;
  L.stages = (smem_limit - fixed) / L.stage_bytes;
  if (L.stages > kTcMaxStages) L.stages = kTcMaxStages;
  L.off_x = L.stages * L.stage_bytes;
  L.off_tab = L.off_x + x_bytes;
  L.off_bar = L.off_tab + tab_bytes;
  L.smem_bytes = L.off_bar + 2 * L.bar_set_bytes;
  return L;
}

// ------------------------------------------------------- weight scales as atoms ----
// w13s [E][2I][H/32] and w2s [E][H][I/32] (row-major E8M0, one byte per 32-element block)
// into the atoms the producer copies per stage: for w13 the tile of a gate/up item (its 64
// gate rows, then its 64 up rows), for w2 the 128 rows of a down item; blocks past the row
// (the second atom of a last half stage) are zero.  One thread per 4-byte word of an atom:
// the word of row m holds blocks 4g..4g+3, 4 bytes of the source row.
__global__ void k_scale_atoms(const uint8_t* __restrict__ w13s, const uint8_t* __restrict__ w2s,
                              uint8_t* __restrict__ w13a, uint8_t* __restrict__ w2a, int E, int H,
                              int I) {
  const int g13 = sf_atoms_per_tile(H), g2 = sf_atoms_per_tile(I);
  const size_t n13 = (size_t)E * (I / 64) * g13 * 128, n2 = (size_t)E * (H / 128) * g2 * 128;
  for (size_t wi = blockIdx.x * (size_t)blockDim.x + threadIdx.x; wi < n13 + n2;
       wi += (size_t)gridDim.x * blockDim.x) {
    const bool up13 = wi < n13;
    const size_t v = up13 ? wi : wi - n13;
    const int pos = (int)(v % 128);       // word within the atom
    const int m = pos / 4 + 32 * (pos % 4);  // byte 4 pos = 16 (m mod 32) + 4 (m / 32)
    const size_t a = v / 128;
    const int ga = up13 ? g13 : g2;
    const int g = (int)(a % ga);
    const size_t tile = a / ga;
    uint32_t word = 0u;
    if (up13) {
      const int t = (int)(tile % (I / 64)), e = (int)(tile / (I / 64));
      const int row = (m < 64) ? 64 * t + m : I + 64 * t + (m - 64);
      if (4 * g < H / 32)
        word = *reinterpret_cast<const uint32_t*>(w13s + ((size_t)e * 2 * I + row) * (H / 32) +
                                                  4 * g);
      reinterpret_cast<uint32_t*>(w13a)[wi] = word;
    } else {
      const int t = (int)(tile % (H / 128)), e = (int)(tile / (H / 128));
      const int row = 128 * t + m;
      if (4 * g < I / 32)
        word = *reinterpret_cast<const uint32_t*>(w2s + ((size_t)e * H + row) * (I / 32) + 4 * g);
      reinterpret_cast<uint32_t*>(w2a)[v] = word;
    }
  }
}

size_t scale_atom_bytes(const Dims& d) {
  return ((size_t)d.E * (d.I / 64) * sf_atoms_per_tile(d.H) +
          (size_t)d.E * (d.H / 128) * sf_atoms_per_tile(d.I)) * 512;
}

cudaError_t launch_scale_atoms(const Dims& d, const Weights& w, uint8_t* atoms, cudaStream_t st) {
  uint8_t* w13a = atoms;
  uint8_t* w2a = atoms + (size_t)d.E * (d.I / 64) * sf_atoms_per_tile(d.H) * 512;
  k_scale_atoms<<<1024, 256, 0, st>>>(w.w13s, w.w2s, w13a, w2a, d.E, d.H, d.I);
  return cudaGetLastError();
}

}  // namespace mtail
