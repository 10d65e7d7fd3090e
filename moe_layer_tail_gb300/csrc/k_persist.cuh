// k_persist.cuh -- the single persistent launch of the tail (defined in k_stream_tc.cu) and
// its grid-wide barrier.
#pragma once

#include <cuda_runtime.h>

#include "moe_tail_internal.cuh"

namespace mtail {

// Grid barrier words: outside every word the call's front clears, never reset between calls.
constexpr int kCtrPersistArrive = 8;
constexpr int kCtrPersistGen = 9;
static_assert(kCtrOutProj < kCtrPersistArrive && kCtrPersistGen < kCtrGUDone &&
                  kCtrPersistGen != kCtrSharedGUDone,
              "the persistent launch's counter words are free");

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide barrier of a launch whose CTAs are all resident: a count of arrivals and a
// generation word; the last CTA to arrive resets the count and advances the generation with
// a release store, the others wait (bounded, acquire) until the generation differs from the
// one they read on arrival.  The generation only grows, so it tags every barrier of every
// call and nothing is reset between calls or graph replays.  False when this CTA's wait
// expired (the status word says so).
__device__ __forceinline__ bool grid_barrier(const Scratch& s, uint64_t budget_ns) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t* arrive = &s.counters[kCtrPersistArrive];
    uint32_t* gen = &s.counters[kCtrPersistGen];
    const uint32_t g0 = ld_acquire_u32(gen);
    __threadfence();  // this CTA's writes (seen by thread 0 through the CTA barrier) first
    int ok = 1;
    if (atomicAdd(arrive, 1u) == gridDim.x - 1) {
      atomicExch(arrive, 0u);
      asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(gen), "r"(g0 + 1u) : "memory");
    } else {
      const uint64_t t0 = globaltimer();
      for (uint32_t i = 1; ld_acquire_u32(gen) == g0; ++i) {
        __nanosleep(32);
        if ((i & 15) == 0 && globaltimer() - t0 > budget_ns) {
          set_status(s.status, kStatusTimeout);
          ok = 0;
          break;
        }
      }
    }
    __threadfence();
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

// The dynamic shared memory the persistent kernel for nmax B columns may take (what its front's
// static shared memory leaves); sets the kernel's attribute.
cudaError_t persistent_smem_limit(int nmax, int* smem_limit);

// Set up the persistent kernel of the handle's layout (its shared-memory size) and return
// how many of its CTAs one SM holds (0: it does not fit).
cudaError_t persistent_prepare(const TcMaps& maps, int* blocks_per_sm);

// The whole call in one cooperative launch of `grid` CTAs (all resident at once); stall:
// CTA 0 leaves at once (failure injection: the others' barrier waits expire); done, seq, ha:
// as for launch_combine (ha also gives x).
cudaError_t launch_persistent(const TcMaps& maps, const Dims& d, const __nv_bfloat16* x,
                              __nv_bfloat16* residual, __nv_bfloat16* out, const Weights& w,
                              const Scratch& s, int grid, uint64_t budget_ns, bool stall,
                              cudaStream_t st, uint32_t* done = nullptr, uint32_t seq = 0u,
                              const HostArgs* ha = nullptr);

// Zero the barrier words of the persistent launch (after a call that gave up on a wait).
cudaError_t persistent_reset(const Scratch& s);

}  // namespace mtail
