// Device helpers shared by the kernels of this library.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gqa_attn.h"

namespace gqa {

__device__ __forceinline__ void report(int32_t* status, int32_t bits) {
  if (status) atomicOr(status, bits);
}

// True when the call's non-finite check found a bad input: every kernel of the
// call then returns at once (skip is the caller's status word, or nullptr when
// the check is off).
__device__ __forceinline__ bool gated_off(const int32_t* skip) {
  return skip && (*reinterpret_cast<const volatile int32_t*>(skip) & ATTN_DEV_NONFINITE);
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

// c * tanh(s / c) written as c * (1 - 2 / (exp(2 s / c) + 1)), evaluated with
// the hardware base-2 exponential. Relative error of the tanh stays near
// fp32 rounding for every |s / c| (the cancellation near 0 costs a few bits
// of a value that is itself small); exp2 overflow to +inf gives exactly c.
__device__ __forceinline__ float softcap_apply(float s, float cap, float two_log2e_over_cap) {
  float e = exp2f(s * two_log2e_over_cap);
  return cap - 2.0f * cap / (e + 1.0f);
}

}  // namespace gqa
