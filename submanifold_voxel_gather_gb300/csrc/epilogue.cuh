// Activation of the fused epilogue (spconv_submconv3d_ex), in fp32.
#pragma once

#include <cuda_runtime.h>

#include "spconv.h"

namespace spconv {

__device__ __forceinline__ float apply_activation(float x, int act) {
  if (act == SPCONV_ACT_RELU) return x > 0.0f ? x : 0.0f;
  if (act == SPCONV_ACT_SILU) return x / (1.0f + expf(-x));
  return x;
}

// Same with the fast exponential and division intrinsics (a few ulp in
// fp32), for results that are rounded to bf16 right after.  For x below
// about -88 the denominator is +inf and the quotient 0 (the limit).
__device__ __forceinline__ float apply_activation_bf16(float x, int act) {
  if (act == SPCONV_ACT_RELU) return x > 0.0f ? x : 0.0f;
  if (act == SPCONV_ACT_SILU) return __fdividef(x, 1.0f + __expf(-x));
  return x;
}

}  // namespace spconv
