// kda_common.cuh -- small device helpers shared by the libkda kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"
#include "kda_internal.h"

namespace kda {

// bf16 bit patterns -> fp32 (exact: a bf16 is the top half of an fp32).
__device__ __forceinline__ float bf16_lo(uint32_t pair) { return __uint_as_float(pair << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t pair) { return __uint_as_float(pair & 0xffff0000u); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
  return x;
}

// 1 / (1 + e^-x) through the correctly rounded reciprocal intrinsic (no
// divide slow path; e^-x = inf gives exactly 0).
__device__ __forceinline__ float sigmoidf_(float x) { return __frcp_rn(1.0f + expf(-x)); }

// log(1 + e^x) without overflow: max(x, 0) + log1p(e^-|x|).
__device__ __forceinline__ float softplusf_(float x) { return fmaxf(x, 0.0f) + log1pf(expf(-fabsf(x))); }

// Programmatic dependent launch.  pdl_wait() returns once the preceding grid
// in the stream has completed and its writes are visible (a no-op when this
// grid was launched normally); pdl_trigger() lets the next grid be scheduled
// before this one finishes.  A kernel may read inputs that no earlier kernel
// of the same call writes before pdl_wait(), and writes nothing before it.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void raise_status(int32_t* status, int32_t bit) {
  if (status != nullptr) atomicOr(status, bit);
}

// Index checks of the debug build (compiled with KDA_DEBUG_BOUNDS=1, the
// library libkda_debugbounds.so): kda_in_bounds(cond, status) is cond, and
// when cond fails it also sets KDA_DEV_BOUNDS, so that the caller skips the
// access it guards.  In every other build it is the constant true and the
// checks compile away.  (compute-sanitizer is not available everywhere these
// kernels run; the debug build is the stand-in.)
#if KDA_DEBUG_BOUNDS
__device__ __forceinline__ bool kda_in_bounds(bool cond, int32_t* status) {
  if (!cond) raise_status(status, KDA_DEV_BOUNDS);
  return cond;
}
#else
__device__ __forceinline__ constexpr bool kda_in_bounds(bool, int32_t*) { return true; }
#endif

}  // namespace kda
