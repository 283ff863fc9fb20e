// Bounded waits shared by the warp-specialised kernels.
#pragma once

#include "common.cuh"
#include "sm100_ptx.cuh"

namespace bd {

constexpr uint64_t kDrainLimitNs = 100000000ull;  // 100 ms for in-flight copies / MMAs at exit

// Wait used at exit to let this CTA's own TMA copies / MMAs finish before its
// shared and tensor memory are released; ignores the abort flag.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > kDrainLimitNs) return false;
  return true;
}

// Single-thread pipeline wait with the kernel-wide limit.
__device__ __forceinline__ bool pipe_wait(uint64_t* bar, uint32_t parity, int* abort_flag, volatile int* gstatus) {
  return mbar_wait(bar, parity, abort_flag, gstatus, kAbortBits, kWaitLimitNs);
}

// Every lane of the warp waits; the result is made warp-uniform so that the
// warp-collective tcgen05.ld / st that follow are executed by all or none.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int* abort_flag, volatile int* gstatus) {
  const bool ok = pipe_wait(bar, parity, abort_flag, gstatus);
  return __all_sync(0xffffffffu, ok);
}

}  // namespace bd
