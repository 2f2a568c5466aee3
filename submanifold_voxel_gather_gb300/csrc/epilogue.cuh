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

// For results that are rounded to bf16 right after: the activation fixed at
// compile time, with the fast exponential and division intrinsics (a few ulp
// in fp32; for x below about -88 the denominator is +inf and the quotient 0,
// the limit), and a dispatcher that runs f(ActTag<act>{}) for a run-time act,
// so that loops over many values test the activation once.
template <int kAct>
struct ActTag {
  static constexpr int value = kAct;
};

template <int kAct>
__device__ __forceinline__ float activation_bf16(float x) {
  if constexpr (kAct == SPCONV_ACT_RELU) return x > 0.0f ? x : 0.0f;
  else if constexpr (kAct == SPCONV_ACT_SILU) return __fdividef(x, 1.0f + __expf(-x));
  else return x;
}

template <typename F>
__device__ __forceinline__ void with_activation(int act, F&& f) {
  if (act == SPCONV_ACT_RELU) f(ActTag<SPCONV_ACT_RELU>{});
  else if (act == SPCONV_ACT_SILU) f(ActTag<SPCONV_ACT_SILU>{});
  else f(ActTag<SPCONV_ACT_NONE>{});
}

}  // namespace spconv
