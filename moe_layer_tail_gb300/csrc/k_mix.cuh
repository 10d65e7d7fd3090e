// k_mix.cuh -- launch plan and launcher of the AttnRes residual mix (k_mix.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace amix {

constexpr int kMaxSources = 32;    // committed blocks + the prefix
constexpr int kMaxThreads = 256;   // per CTA
constexpr int kMaxCluster = 8;     // CTAs per row (portable cluster size)
constexpr int kMaxRows = 4096;
constexpr int kMaxHidden = 1 << 16;

struct MixPlan {
  int C;         // CTAs per row, one thread-block cluster
  int W;         // columns per CTA (hidden / C, a multiple of 8)
  int threads;   // per CTA
  size_t smem;   // dynamic shared memory per CTA
  int reg_smax;  // > 0: the register kernel for up to this many sources; 0: the staged one
};

// The plan for `hidden` columns and S sources; false when the shape is not supported
// (hidden not a multiple of 8 in [8, 65536], S outside [1, 32], or staging too large).
bool mix_plan(int hidden, int S, MixPlan* p);

struct MixArgs {
  const uint16_t* sub;     // [R, H] bf16
  uint16_t* prefix;        // [R, H] bf16, in/out
  uint16_t* blocks;        // [n_blocks + commit, R, H] bf16
  const uint16_t* q;       // [H] bf16
  const uint16_t* gamma;   // [H] bf16
  uint16_t* mix;           // [R, H] bf16, out
  uint16_t* y;             // [R, H] bf16, out
  int R, H, n_blocks, commit;
  float eps;
  int debug_stall;         // one CTA waits for a value that never comes (failure test)
};

cudaError_t launch_attnres_mix(const MixArgs& a, const MixPlan& p, cudaStream_t st, bool pdl);

// The device status word of the mix (synchronous copy); clear: zero it afterwards.
cudaError_t mix_status(int* out, bool clear);

}  // namespace amix
