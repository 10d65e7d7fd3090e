// moe_tail_internal.cuh -- device helpers, scratch layout and launcher declarations shared
// by the kernels of libmoe_tail.so.  Nothing here is part of the public C ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace mtail {

// Hard limits (checked at create time).  The default (tcgen05) form takes up to 32 rows (the
// top-k dedup keeps each expert's users as a 32-bit row mask); the other expert forms, the
// fused front, the persistent launch and the routing without allocation keep per-row
// register arrays of 16.
constexpr int kMaxRows = 32;
constexpr int kMaxRowsOther = 16;
constexpr int kMaxTopK = 32;
constexpr int kMaxExperts = 1024;
// dynamic shared memory a streaming CTA may take (the opt-in maximum per block)
constexpr int kSmemLimit = 232448;
// parts a row's add + RMSNorm may be split into (the persistent launch; H / 256 at most)
constexpr int kMaxNormParts = 128;
constexpr int kMaxPicks = kMaxRows * kMaxTopK;  // (row, slot) pairs of one call
constexpr int kMaxOutProjParts = 8;  // K parts of an out_proj box at most
// A shared-expert gate/up item (64 gate + 64 up rows over all of H) may be split along K into
// up to kMaxSharedParts parts when it is larger than an SM's share of the launch or when the
// shared items are too few to keep most SMs streaming before the routing is known (the
// tensor-core form), for shared experts of at most kMaxSharedSplitItems items.
constexpr int kMaxSharedParts = 4;
constexpr int kMaxSharedSplitItems = 256;

// Device status word bits (sticky; read by moe_tail_get_status; the same values as
// MOE_TAIL_STATUS_* in moe_tail.h).
enum : int32_t {
  kStatusBadRouting = 1 << 0,   // top-k found only NaN logits left for a pick
  kStatusBadDistinct = 1 << 1,  // distinct-expert count out of range
  kStatusTimeout = 1 << 2,      // a bounded wait expired
  kStatusBadTile = 1 << 3,      // a work item outside its matrix was skipped
};

struct Dims {
  int R;        // rows of this call
  int Rmax;     // rows the handle was created for (height of the activation boxes)
  int H, E, k, I, Is;
  int Ha;       // attention out_proj K (0: none)
  int Pk;       // K parts of an out_proj box (1: the launch writes x itself)
  float eps;
  int sparts = 1;  // K parts of a shared-expert gate/up item (tensor-core gate/up roles)
};

// The buffers and number of one host-buffer call (moe_tail_run_host), in page-locked memory
// mapped into the device's address space: the kernels that read or write the call's buffers
// take them from here at run time, so one captured graph serves every call.
struct HostArgs {
  const void* x;
  void* residual;
  void* out;
  uint32_t seq;  // the value the call's last kernel writes to the completion word
  uint32_t pad;
};
__device__ __forceinline__ const void* ha_ptr(const void* const* p) {
  return reinterpret_cast<const void*>(
      *reinterpret_cast<const volatile unsigned long long*>(p));
}

struct Weights {
  const __nv_bfloat16* gamma;
  const __nv_bfloat16* w_r;
  const uint8_t* w13c;
  const uint8_t* w13s;
  const uint8_t* w2c;
  const uint8_t* w2s;
  const __nv_bfloat16* ws13;
  const __nv_bfloat16* ws2;
  const __nv_bfloat16* wsg;  // shared-expert gate [H], or null
  const __nv_bfloat16* wo;   // attention out_proj [H, Ha], or null
  // the tensor-core form's copies of w13s and w2s in scale-factor atoms (sf_atom_offset):
  // w13a [E][I/64 items][H/128 atoms][512 B] (an item's 64 gate rows, then its 64 up rows),
  // w2a [E][H/128 items][2 ceil(I/256) atoms][512 B]; null in the other forms
  const uint8_t* w13a;
  const uint8_t* w2a;
};

// Every buffer a call needs, carved from one allocation made at create time.
struct Scratch {
  __nv_bfloat16* rnew;   // [Rmax, H] bf16(x + residual), copied to the residual at the end
  __nv_bfloat16* n;      // [Rmax, H] normalised activations (bf16)
  __half* n16;           // [Rmax, H] n as f16, scaled by 2^-p per row
  float* n16s;           // [Rmax] the 2^p of each row
  float* logits;         // [Rmax, E]
  float* logit_parts;    // [16, Rmax, E] router partial sums over K parts
  int32_t* ids;          // [Rmax, k] picks in pick order
  float* wts;            // [Rmax, k]
  int32_t* n_distinct;   // [1]
  int32_t* uniq;         // [Rmax*k] distinct expert ids, ascending
  int32_t* user_off;     // [Rmax*k + 1] CSR offsets into user_list
  int32_t* user_list;    // [Rmax*k] pick indices r*k + slot, in (r, slot) order
  __nv_bfloat16* mid;    // [Rmax*k, I] SiLU(gate)*up of each pick (bf16)
  __half* mid16;         // [Rmax*k, I] mid as f16 (unscaled, or scaled by 2^-p per 32-element
                         // block where its largest magnitude leaves [2^-10, 2^15));
                         // row = the pick's position in user_list (users of an expert adjacent)
  float* mid16s;         // [Rmax*k, I/32] the 2^p of each block, same rows
  __nv_bfloat16* ms;     // [Rmax, Is] shared-expert intermediate (bf16)
  float* y;              // [Rmax*k, H] routed expert outputs
  float* ys;             // [Rmax, H] shared expert output
  float* sgate;          // [Rmax] sigmoid gate of the shared output (when a gate is given)
  float* gate_part;      // [Rmax, kMaxNormParts] the persistent launch's per-part gate logits
  __nv_bfloat16* xproj;  // [Rmax, H] x = out_proj(attn) for moe_tail_run_attn (one K part)
  float* xpart;          // [kMaxOutProjParts, Rmax, H] fp32 sums of each out_proj K part
  float* gpart;          // [kMaxSharedSplitItems, kMaxSharedParts, 128, Rmax] fp32 sums of the
                         // K parts of split shared gate/up items (rows: 64 gate, 64 up)
  uint8_t* np4;          // [4 Rmax, H/2] E2M1 planes of n (row 4r + p = plane p of row r)
  uint8_t* np4a;         // [H/128][512] their E8M0 scales in scale-factor atoms (row 4r + p)
  uint8_t* mid4;         // [4 Rmax k, I/2] E2M1 planes of mid (row 4 slot + p, slot = the
                         // pick's position in user_list)
  uint8_t* mid4a;        // [min(E, Rmax k)][2 ceil(I/256)][512] their E8M0 scales in
                         // scale-factor atoms per distinct expert (row 4 (slot - u0) + p)
  unsigned long long* tl;  // [kTlSlots] %globaltimer stamps of the last run, or null (the
                           // timeline debug flag off)
  int32_t* status;       // [1] sticky device status word
  uint32_t* counters;    // [kCtrWords] work counters, tickets and per-expert progress
};

// Debug bits the kernels read (same values as MOE_TAIL_DEBUG_* in moe_tail.h).
constexpr uint32_t kDebugStallFirstStage = 4u;
constexpr uint32_t kDebugMmaSync = 16u;
constexpr uint32_t kDebugTimeline = 32u;

// Timeline slots (same order as MOE_TAIL_TL_* in moe_tail.h): the first or last %globaltimer
// reading of each milestone of a run, recorded when the handle has a timeline buffer.
enum : int {
  kTlNormStart = 0,   // norm launch: first CTA past its wait on the previous launch
  kTlNormEnd,         // norm launch: last CTA done
  kTlRouterStart,     // router launch: first CTA past its wait
  kTlTopkStart,       // router launch: its last CTA starts top-k and the dedup
  kTlRouted,          // router launch: routing published
  kTlGateUpStart,     // gate/up launch: first CTA entered
  kTlGateUpFirstCopy, // gate/up launch: first weight copy issued
  kTlGateUpRouted,    // gate/up launch: first routed expert's weight copy issued
  kTlGateUpEnd,       // gate/up launch: last CTA done
  kTlDownStart,       // down launch: first CTA entered
  kTlDownFirstCopy,   // down launch: first weight copy issued
  kTlDownEnd,         // down launch: last CTA done
  kTlCombineStart,    // combine launch: first CTA entered
  kTlCombineEnd,      // combine launch: last output written
  kTlRouterAllStarted,  // router launch: last CTA past its wait
  kTlGateUpAllCopying,  // gate/up launch: last CTA's first weight copy issued
  kTlSlots
};

// counters[] words (all zeroed at the start of every call by the front)
enum : int {
  kCtrGateUp = 0,        // next work item of the gate/up launch
  kCtrDown = 1,          // next work item of the down launch
  kCtrFrontTicket = 2,   // router CTAs done (the last one ranks the experts)
  kCtrRouted = 3,        // nonzero once the call's routing tables are written (release)
  kCtrSharedGUDone = 4,  // shared-expert gate/up items finished
  kCtrGUAllDone = 5,     // gate/up items finished, shared and routed together (release)
  kCtrCombineTicket = 10,  // combine CTAs done (the last one signals a host-visible word)
  kCtrGUDone = 16,       // [kMaxPicks] routed gate/up items finished, per distinct expert
  kCtrMidFlag = 16 + kMaxPicks,  // [kMaxPicks] nonzero: some 32-block of the expert's mid
                                 // carries a power-of-two scale
  kCtrOutProj = 6,       // next work item of the out_proj launch (runs before the norm
                         // launch, which zeroes it with the rest for the next call)
  kCtrTileDone = 16 + 2 * kMaxPicks,  // [256] down items finished per 128 hidden outputs
  kCtrSharedParts = 16 + 2 * kMaxPicks + 256,  // [kMaxSharedSplitItems] K parts of a split
                                               // shared gate/up item finished
  kCtrWords = 16 + 2 * kMaxPicks + 256 + 256
};

// ------------------------------------------------------------------ device helpers ----

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Four bytes of packed E2M1 pairs -> four f16x2 registers (element 2j in the low half).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t& h0, uint32_t& h1,
                                                uint32_t& h2, uint32_t& h3) {
  asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %4;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0;\n cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      " cvt.rn.f16x2.e2m1x2 %2, b2;\n cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
      : "r"(w));
}

// E8M0 scale byte -> float 2^(s-127) (s = 0 gives the subnormal 2^-127; 255 is not used).
__device__ __forceinline__ float e8m0_to_float(uint32_t s) {
  return s ? __uint_as_float(s << 23) : __uint_as_float(0x00400000u);
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait until *p >= need (acquire at GPU scope): false when the budget ran out.
__device__ __forceinline__ bool wait_count(const uint32_t* p, uint32_t need, uint64_t budget_ns,
                                           uint32_t sleep_ns = 64) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  if (v >= need) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    __nanosleep(sleep_ns);
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    if (v >= need) return true;
    if ((i & 15) == 0 && globaltimer() - t0 > budget_ns) return false;
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// SiLU in fp32 with the fast exponential and division (a few ulp; mid is rounded to bf16
// right after).
__device__ __forceinline__ float silu_f(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// 2^e as a float, exact for e in [-127, 127] (2^-127 is the subnormal 0x00400000).
__device__ __forceinline__ float exp2_int(int e) {
  return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// E2M1 activation planes (the tensor-core form of the routed experts).  A block of 32 values
// becomes the sum of four planes, each an E2M1 code per value times one power of two 2^e per
// plane: e is the smallest exponent with amax <= 6 * 2^e for the block's largest magnitude
// amax of what the planes before it left over (-127 when that is zero), the codes are the
// nearest E2M1 values (ties to even) of value / 2^e.
__device__ __forceinline__ int e2m1_plane_exp(float amax) {
  if (!(amax > 0.f)) return -127;
  const uint32_t b = __float_as_uint(amax);
  const int E = (int)((b >> 23) & 0xFF) - 127;
  if (E < -126) return -127;  // subnormal: amax / 2^-127 < 2
  const int e = E - 2 + ((b & 0x7FFFFFu) > 0x400000u ? 1 : 0);
  return e > 127 ? 127 : e;
}

// Nearest E2M1 code of x (ties to even, saturating at 6), in the low nibble.
__device__ __forceinline__ uint32_t e2m1_code(float x) {
  uint32_t w;
  asm("{ .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n mov.b32 %0, {t, t, t, t}; }"
      : "=r"(w)
      : "f"(0.f), "f"(x));
  return w & 0xFu;
}

// Eight values -> eight E2M1 codes in one word (value 2j in the low nibble of byte j).
__device__ __forceinline__ uint32_t e2m1x8_pack(const float (&x)[8]) {
  uint32_t w;
  asm("{ .reg .b8 b0, b1, b2, b3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      " mov.b32 %0, {b0, b1, b2, b3}; }"
      : "=r"(w)
      : "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]), "f"(x[7]));
  return w;
}

// Scale-factor atoms: the layout in which tcgen05.cp (32 rows x 128 bits, copied to all four
// lane quadrants) brings E8M0 scales into tensor memory for the block-scaled MMAs.  One atom
// of 512 bytes holds 4 consecutive 32-element blocks of 128 operand rows, row m's block b at
// byte 16 (m mod 32) + 4 (m / 32) + b; consecutive atoms cover consecutive groups of 4
// blocks.  Byte offset of (row, block) for a 128-row operand tile, block counted from 0:
__host__ __device__ __forceinline__ uint32_t sf_atom_offset(int row, int block) {
  return 512u * (uint32_t)(block >> 2) + 16u * (uint32_t)(row & 31) + 4u * (uint32_t)(row >> 5) +
         (uint32_t)(block & 3);
}
// atoms of one operand tile over K elements (whole 256-element stages: two atoms each)
__host__ __device__ __forceinline__ int sf_atoms_per_tile(int K) { return 2 * ((K + 255) / 256); }

// Value of the E2M1 code in the low nibble of `code`.
__device__ __forceinline__ float e2m1_value(uint32_t code) {
  uint32_t h;
  asm("{ .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n"
      " cvt.rn.f16x2.e2m1x2 %0, b0; }"
      : "=r"(h)
      : "r"(code & 0xFu));
  return __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
}

// Timeline stamps (only when the handle records a timeline): the first reading of a slot
// (the word is zero until then), or the latest.
__device__ __forceinline__ void tl_first(unsigned long long* tl, int slot) {
  if (tl) atomicCAS(tl + slot, 0ull, (unsigned long long)globaltimer());
}
__device__ __forceinline__ void tl_last(unsigned long long* tl, int slot) {
  if (tl) atomicMax(tl + slot, (unsigned long long)globaltimer());
}

__device__ __forceinline__ void set_status(int32_t* status, int32_t bit) {
  atomicOr(reinterpret_cast<int*>(status), bit);
}

// Programmatic dependent launch: wait until the previous kernel in the stream has completed
// and its writes are visible (a no-op when the launch was not programmatic), and let the
// next kernel's CTAs start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch `kernel` on `st`, optionally as a programmatic dependent launch.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t st, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Shared-memory plan of the streaming kernels for one handle (depends on its row count).
constexpr int kMaxStreamStages = 8;
struct StreamLayout {
  int stages;       // pipeline stages (<= kMaxStreamStages)
  int stage_bytes;  // 16 KB weight tile + act_rows x 512 B of activations
  int act_rows;     // activation rows a stage holds: 4, 8 or 16
  int win_bytes;    // one scale window: 8 KB weight scales + act_rows x 256 B
  int nt_max;       // N-tiles of 8 users (1 or 2)
  int off_win, off_red, off_tab, off_bar;  // byte offsets of the regions after the stages
  int smem_bytes;   // dynamic shared memory of a launch
  int tab_picks;    // entries of the dedup tables (rows x k of the handle)
};

// TMA descriptors of the streamed matrices (built once at create time) and the plan.
struct StreamMaps {
  CUtensorMap w13;        // u8 [E*2I, H/2], box {128 B, 64 rows}, 128-byte swizzle
  CUtensorMap w2;         // u8 [E*H, I/2], box {128 B, 128 rows}, 128-byte swizzle
  CUtensorMap ws13;       // bf16 [2Is, H], box {64, 64}, 128-byte swizzle
  CUtensorMap ws2;        // bf16 [H, Is], box {64, 128}, 128-byte swizzle
  CUtensorMap n;          // bf16 [Rmax, H] scratch n, box {64, Rmax}, 128-byte swizzle
  CUtensorMap ms;         // bf16 [Rmax, Is] scratch ms, box {64, Rmax}, 128-byte swizzle
  CUtensorMap n16;        // f16 [Rmax, H] scratch n16, box {256, Rmax}
  CUtensorMap mid16[3];   // f16 [Rmax*k, I] scratch mid16, box {256, 4 / 8 / 16 rows}
  CUtensorMap mid16s[3];  // f32 [Rmax*k, I/32], box {min(64, I/32), 4 / 8 / 16 rows}
  CUtensorMap w13s;       // u8 [E*2I, H/32], box {64 B, 64 rows} (H > 2048 only)
  CUtensorMap w2s;        // u8 [E*H, I/32], box {64 B, 128 rows} (I > 2048 only)
  CUtensorMap wo;         // bf16 [H, Ha], box {64, 128}, 128-byte swizzle (Ha > 0 only)
  CUtensorMap attn;       // bf16 [rows, Ha] of the call, box {64, Rmax}, 128-byte swizzle
  StreamLayout lay;
};

// Shared-memory plan of the tensor-core streaming kernels (depends on the handle's rows).
struct TcLayout {
  int nmax;         // B columns of an item at most: 4 planes x rows (16, 32, 64 or 128)
  int aslots;       // accumulator slots (2, or 1 at 128 columns: tensor memory holds 512)
  int b_bytes;      // activation tile of a stage: nmax rows x 128 bytes
  int stage_bytes;  // 16 KB weights + b_bytes + 2 KB scale-factor atoms
  int stages;
  int off_x, off_tab, off_bar, smem_bytes;
  int bar_set_bytes;  // one set of barriers and item words (two sets follow off_bar)
  int tab_picks;    // entries of the dedup tables (rows x k of the handle)
};

// TMA descriptors of the tensor-core streaming kernels.
struct TcMaps {
  CUtensorMap w13;        // u8 [2E][I][H/2] (rows (2e + half) I + j), box {128 B, 64, 2}:
                          // a stage's 64 gate and 64 up rows in one copy, 128-byte swizzle
  CUtensorMap ws13;       // bf16 [2][Is][H], box {64, 64, 2}, 128-byte swizzle
  CUtensorMap w2, ws2, n, ms;  // as in StreamMaps
  CUtensorMap np4;        // u8 [4 Rmax, H/2] planes of n, box {128 B, nmax}, 128-byte swizzle
  CUtensorMap mid4[4];    // u8 [4 P, I/2], box {128 B, 16 / 32 / 64 / 128 rows}, 128-byte swizzle
  TcLayout lay;
};

// ------------------------------------------------------------------ launchers ----
// Each returns the cudaError_t of its launch.

// ha: take x and residual from a host-buffer call's arguments instead (null: as given)
cudaError_t launch_add_rmsnorm(const Dims& d, const __nv_bfloat16* x,
                               const __nv_bfloat16* residual, const Weights& w,
                               const Scratch& s, cudaStream_t st, bool pdl,
                               const float* xpart = nullptr, bool planes = false,
                               const HostArgs* ha = nullptr);
cudaError_t launch_router(const Dims& d, const Weights& w, const Scratch& s, cudaStream_t st,
                          bool pdl);
cudaError_t launch_topk_dedup(const Dims& d, const Scratch& s, cudaStream_t st, bool pdl);
cudaError_t launch_router_topk(const Dims& d, const Weights& w, const Scratch& s,
                               cudaStream_t st, bool pdl);
cudaError_t launch_front_fused(const Dims& d, const __nv_bfloat16* x,
                               const __nv_bfloat16* residual, const Weights& w, const Scratch& s,
                               cudaStream_t st, bool pdl);
cudaError_t launch_experts_simple(const Dims& d, const Weights& w, const Scratch& s,
                                  int num_sms, cudaStream_t st);
int make_stream_maps(StreamMaps* out, const Dims& d, const Weights& w, const Scratch& s);
// The call's attention-output map (bf16 [rows, Ha] at attn): 0, or -1/-2 as make_stream_maps.
int make_attn_map(StreamMaps* m, const void* attn, int rows, const Dims& d);
StreamLayout make_stream_layout(int Rmax, int k);
cudaError_t prepare_stream_kernels();
cudaError_t prepare_front_kernels();
int router_max_parts();
cudaError_t launch_stream(int phase, const StreamMaps& maps, const Dims& d, const Weights& w,
                          const Scratch& s, int num_sms, uint64_t budget_ns, cudaStream_t st,
                          bool pdl, uint32_t debug);
// smem_limit: the dynamic shared memory the kernel may take (less for the persistent one,
// whose front keeps static shared memory)
TcLayout make_tc_layout(int Rmax, int k, int smem_limit);
int make_tc_maps(TcMaps* out, const StreamMaps& sm, const Dims& d, const Weights& w,
                 const Scratch& s, int smem_limit);
cudaError_t prepare_stream_tc_kernels();
cudaError_t launch_stream_tc(int phase, const TcMaps& maps, const Dims& d, const Weights& w,
                             const Scratch& s, int num_sms, uint64_t budget_ns, cudaStream_t st,
                             bool pdl, uint32_t debug);
// The router's parts (k_front.cu): 16-expert tiles x K parts of plen elements, the shared
// memory of one part for `warps` warps and the offset of its reduction tiles in it.
struct RouterPlan {
  int tiles, parts, plen, red_off;
  size_t smem;
};
RouterPlan router_plan(int R, int H, int E, int warps);

// bytes of the two atom copies (w13a then w2a) and the launch that writes them from w13s, w2s
size_t scale_atom_bytes(const Dims& d);
cudaError_t launch_scale_atoms(const Dims& d, const Weights& w, uint8_t* atoms, cudaStream_t st);
// done: a host-visible word the call's last combine CTA sets to seq once every output is
// visible to the host (null: none); ha: take out, residual and seq from a host-buffer call's
// arguments instead (null: as given); down_grid: the tensor-core down launch's grid, whose
// items the combine waits to see all claimed before its per-tile waits (0: no such wait)
cudaError_t launch_combine(const Dims& d, const Scratch& s, __nv_bfloat16* out,
                           __nv_bfloat16* residual, cudaStream_t st, bool pdl, bool wait_tiles,
                           uint64_t budget_ns, bool gated, uint32_t* done = nullptr,
                           uint32_t seq = 0u, const HostArgs* ha = nullptr, int down_grid = 0);

}  // namespace mtail
