// k_persist.cuh -- the single persistent launch of the tail (defined in k_simple.cu).
#pragma once

#include <cuda_runtime.h>

#include "moe_tail_internal.cuh"

namespace mtail {

// CTAs of the persistent launch that one SM can hold (0: the kernel does not fit).
cudaError_t persistent_blocks_per_sm(int* blocks);

// The whole call in one cooperative launch of `grid` CTAs (all resident at once); stall:
// CTA 0 skips the barriers (failure injection: the others' waits expire).
cudaError_t launch_persistent(const Dims& d, const __nv_bfloat16* x,
                              const __nv_bfloat16* residual_in, __nv_bfloat16* residual,
                              __nv_bfloat16* out, const Weights& w, const Scratch& s, int grid,
                              uint64_t budget_ns, bool stall, cudaStream_t st);

// Zero the barrier words of the persistent launch (after a call that gave up on a wait).
cudaError_t persistent_reset(const Scratch& s);

}  // namespace mtail
