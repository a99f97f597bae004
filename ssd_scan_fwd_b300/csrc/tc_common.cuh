// tc_common.cuh -- small device helpers shared by the non-persistent
// tensor-core kernels (chunk states, chunk outputs, per-chunk gradients).
#pragma once

#include <cstdint>

#include "sm100.cuh"

namespace ssd {
namespace tc {

constexpr float kLog2e = 1.4426950408889634f;

// 2^x by the hardware's approximate base-2 exponential (PTX ex2.approx).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// mbarrier wait with a 2 s limit on the global timer; false when it ran out.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = sm100::globaltimer_ns();
  while (!sm100::mbar_try_wait(bar, parity)) {
    if (sm100::globaltimer_ns() - t0 > 2000000000ull) return false;
  }
  return true;
}

// K-major operand with K spread over 64-element column blocks of `blk` bytes
// (128-byte swizzle): descriptor start-address step (16-byte units) of K
// step kk (16 elements).
__device__ __forceinline__ uint64_t kstep_cols(uint32_t kk, uint32_t blk) {
  return (uint64_t)((kk >> 2) * (blk >> 4) + (kk & 3u) * 2u);
}

// Sixteen zero columns into TMEM (this warp's 32 lanes).
__device__ __forceinline__ void tmem_zero16(uint32_t taddr) {
  uint32_t z[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) z[i] = 0u;
  sm100::tmem_st16(taddr, z);
}

}  // namespace tc
}  // namespace ssd
