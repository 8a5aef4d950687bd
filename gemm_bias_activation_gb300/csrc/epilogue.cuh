// Epilogue activations, applied in fp32 to z = accumulator + bias.
//
// GELU uses the exact erf form (the "Coalesce" README, "Notes for future
// sessions": erff, not the tanh approximation).  Softplus is log(1 + e^z)
// with beta = 1 (the "MLP Megakernel" README, "Architecture"), evaluated as
// max(z, 0) + log1p(exp(-|z|)), which cannot overflow.
#pragma once

#include <math.h>

namespace coalesce {

enum ActKind : int { kActNone = 0, kActRelu = 1, kActGeluErf = 2, kActSoftplus = 3 };

__device__ __forceinline__ float act_relu(float z) { return fmaxf(z, 0.0f); }

__device__ __forceinline__ float act_gelu_erf(float z) {
  return 0.5f * z * (1.0f + erff(z * 0.70710678118654752f));
}

__device__ __forceinline__ float act_softplus(float z) {
  return fmaxf(z, 0.0f) + log1pf(expf(-fabsf(z)));
}

template <int kAct>
__device__ __forceinline__ float act_apply(float z) {
  if constexpr (kAct == kActRelu) {
    return act_relu(z);
  } else if constexpr (kAct == kActGeluErf) {
    return act_gelu_erf(z);
  } else if constexpr (kAct == kActSoftplus) {
    return act_softplus(z);
  } else {
    return z;
  }
}

}  // namespace coalesce
