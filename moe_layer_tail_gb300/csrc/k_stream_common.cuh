// k_stream_common.cuh -- pieces shared by the two forms of the weight-streaming expert
// kernels (k_stream.cu: CUDA-core dequantisation into mma.sync; k_stream_tc.cu: tcgen05
// block-scaled MMAs): stage geometry, the work-item list of a launch, and PTX wrappers for
// mbarriers and TMA.  Internal to libmoe_tail.so.
#pragma once

#include "moe_tail_internal.cuh"

namespace mtail {

constexpr int kChunkF4 = 256;     // MXFP4 elements per stage row (128 bytes)
constexpr int kChunkBF = 64;      // bf16 elements per stage row (128 bytes)
constexpr int kStageW = 16384;    // 128 weight rows x 128 bytes
constexpr int kWinK = 2048;       // K elements per scale window
constexpr int kWinStages = kWinK / kChunkF4;
constexpr int kWinW = 8192;       // weight scales of one window: 128 rows x 64 bytes

enum : int { kSharedGU = 0, kRoutedGU = 1, kSharedDN = 2, kRoutedDN = 3, kOutProj = 4 };

struct Item {
  int kind;
  int d;           // routed: the expert's distinct slot (else -1)
  int row0, row1;  // tensor-map rows: gate (or single) box, up box
  int out0;        // first output index (j for gate/up, h for down)
  int k0, K, nst;  // first K element (out_proj parts), K elements and stages of the item
  int part;        // out_proj: K part of its 128-output box
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

// Launches: 0 = gate/up, 1 = down, 2 = the attention out_proj in front of the tail.
__device__ __forceinline__ int items_of(int phase, const Dims& dm, int D) {
  return (phase == 0) ? dm.Is / 64 + D * (dm.I / 64)
         : (phase == 1) ? dm.H / 128 + D * (dm.H / 128)
                        : (dm.H / 128) * dm.Pk;
}

__device__ __forceinline__ int work_counter(int phase) {
  return (phase == 0) ? kCtrGateUp : (phase == 1) ? kCtrDown : kCtrOutProj;
}

__device__ __forceinline__ Item decode_item(int phase, int item, const Dims& dm,
                                            const Tables& s, int D) {
  Item it;
  it.u0 = 0;
  it.row1 = 0;
  it.d = -1;
  it.k0 = 0;
  it.part = 0;
  if (phase == 0) {
    const int ns = dm.Is / 64;
    it.K = dm.H;
    if (item < ns) {
      it.kind = kSharedGU;
      it.out0 = item * 64;
      it.row0 = it.out0;
      it.row1 = dm.Is + it.out0;
      it.U = dm.R;
      it.nst = (dm.H + kChunkBF - 1) / kChunkBF;
    } else {
      const int q = item - ns, per = dm.I / 64;
      const int d = min(q / per, D - 1);
      const int e = s.uniq[d];
      it.kind = kRoutedGU;
      it.d = d;
      it.out0 = (q % per) * 64;
      it.row0 = e * 2 * dm.I + it.out0;
      it.row1 = it.row0 + dm.I;
      it.u0 = s.off[d];
      it.U = s.off[d + 1] - it.u0;
      it.nst = (dm.H + kChunkF4 - 1) / kChunkF4;
    }
  } else if (phase == 2) {
    // out_proj: 128 rows of W_o (hidden outputs), one of Pk K parts, against every row's
    // attention output
    it.kind = kOutProj;
    it.part = item % dm.Pk;
    it.K = dm.Ha / dm.Pk;  // a multiple of 64
    it.k0 = it.part * it.K;
    it.out0 = (item / dm.Pk) * 128;
    it.row0 = it.out0;
    it.U = dm.R;
    it.nst = it.K / kChunkBF;
  } else {
    const int ns = dm.H / 128;
    if (item < ns) {
      it.kind = kSharedDN;
      it.K = dm.Is;
      it.out0 = item * 128;
      it.row0 = it.out0;
      it.U = dm.R;
      it.nst = (dm.Is + kChunkBF - 1) / kChunkBF;
    } else {
      const int q = item - ns, per = dm.H / 128;
      const int d = min(q / per, D - 1);
      const int e = s.uniq[d];
      it.kind = kRoutedDN;
      it.d = d;
      it.K = dm.I;
      it.out0 = (q % per) * 128;
      it.row0 = e * dm.H + it.out0;
      it.u0 = s.off[d];
      it.U = s.off[d + 1] - it.u0;
      it.nst = (dm.I + kChunkF4 - 1) / kChunkF4;
    }
  }
  it.U = max(1, min(it.U, kMaxRows));
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
__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
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
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(policy)
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
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
      "%2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void mma_f16(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// Four 8x8 b16 matrices from shared memory: lane i gives the address of row i & 7 of matrix
// i >> 3; lane l receives word l & 3 of row l >> 2 of each matrix.
__device__ __forceinline__ void ldsm_x4(const void* p, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
// d = A * B for one m16n8k16 f16 product (no accumulator input).
__device__ __forceinline__ void mma_f16_z(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%10,%10,%10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}
__device__ __forceinline__ void mma_bf16(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Byte offset of 16-byte chunk c of row r in a box of 128-byte rows written by TMA with the
// 128-byte swizzle (chunk index XOR the row's low 3 bits; box base 1024-byte aligned).
__device__ __forceinline__ int swz128_off(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

// E8M0 byte i of a little-endian word of four scales -> float 2^(s-127); the byte 0
// (2^-127) flushes to 0.
__device__ __forceinline__ float e8m0_byte(uint32_t w, int i) {
  return __uint_as_float((i < 3 ? (w << (23 - 8 * i)) : (w >> 1)) & 0x7F800000u);
}

}  // namespace mtail
