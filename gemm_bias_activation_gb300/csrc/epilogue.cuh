// Epilogue activations, applied in fp32 to z = accumulator + bias.
//
// GELU uses the exact erf form (the "Coalesce" README, "Notes for future
// sessions": erff, not the tanh approximation).  Softplus is log(1 + e^z)
// with beta = 1 (the "MLP Megakernel" README, "Architecture"), evaluated as
// max(z, 0) + log1p(exp(-|z|)), which cannot overflow.
#pragma once

#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

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
__device__ __forceinline__ float act_apply(float z);

// Softplus for 16-bit results: the same identity with the special-function
// unit's exponential and logarithm (__expf, __logf).  For z <= 0 terms,
// 1 + e^-|z| lies in (1, 2], where __logf's absolute error is below 2^-21;
// with __expf's relative error the result is within ~1e-6 of softplus(z),
// far below half an ulp of any fp16/bf16 value it is rounded to.
__device__ __forceinline__ float act_softplus_fast(float z) {
  return fmaxf(z, 0.0f) + __logf(1.0f + __expf(-fabsf(z)));
}

// act_apply for results that are rounded to fp16/bf16 next: softplus takes
// the fast form above, the others are unchanged.
template <int kAct>
__device__ __forceinline__ float act_apply_16(float z) {
  if constexpr (kAct == kActSoftplus) {
    return act_softplus_fast(z);
  } else {
    return act_apply<kAct>(z);
  }
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

// ---------------------------------------------------------------------------
// Softplus on packed fp16 pairs, for the chained MLP whose activations are
// fp16 tensor-core operands anyway.
//
//   softplus(z) = max(z, 0) + log1p(t),   t = exp(-|z|) = 2^(-|z| log2 e) in (0, 1]
//
// t comes from one ex2.approx.f16x2 (special-function unit, two values per
// operation); log1p(t) on [0, 1] is the polynomial t (c1 + c2 t + c3 t^2),
// whose coefficients are a minimax fit made for this library with Lawson's
// algorithm (iteratively reweighted least squares) on 20001 points of [0, 1]:
// max |error| 5.3e-4 in exact arithmetic, 6.9e-4 with the coefficients
// rounded to fp16.  Everything is evaluated in fp16x2 (Horner with fused
// multiply-adds): six instructions per pair of values, the |z| folding into
// the multiply.  Against the fp64 definition this keeps a single softplus
// within 2e-3 + 2^-10 |ref| and the chained workloads within ~4e-3 of the
// oracle (tolerance 1e-2).
// ---------------------------------------------------------------------------
// fp16 bit patterns, duplicated into both halves: -log2(e) and the three
// polynomial coefficients 0.98745419, -0.40841109, 0.11463896 (rounded to
// fp16: 0.98730469, -0.40844727, 0.11462402).
constexpr uint32_t kNegLog2eX2 = 0xBDC5BDC5u;
constexpr uint32_t kLog1pC1X2 = 0x3BE63BE6u;
constexpr uint32_t kLog1pC2X2 = 0xB689B689u;
constexpr uint32_t kLog1pC3X2 = 0x2F562F56u;

__device__ __forceinline__ uint32_t softplus_f16x2(uint32_t z) {
  const uint32_t neg_log2e = kNegLog2eX2;
  const uint32_t c1 = kLog1pC1X2;
  const uint32_t c2 = kLog1pC2X2;
  const uint32_t c3 = kLog1pC3X2;
  uint32_t a, e, t, q, r, h;
  asm("abs.f16x2 %0, %1;" : "=r"(a) : "r"(z));  // folds into the multiply below
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(e) : "r"(a), "r"(neg_log2e));
  asm("ex2.approx.f16x2 %0, %1;" : "=r"(t) : "r"(e));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(q) : "r"(c3), "r"(t), "r"(c2));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(q) : "r"(q), "r"(t), "r"(c1));
  asm("max.f16x2 %0, %1, %2;" : "=r"(r) : "r"(z), "r"(0u));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(h) : "r"(q), "r"(t), "r"(r));
  return h;
}

// ---------------------------------------------------------------------------
// The same softplus with its argument and result in log2 units, for a chain
// that carries its activations scaled by log2(e):
//
//   z' = z log2 e,   h' = softplus(z) log2 e = max(z', 0) + log2(1 + t),  t = 2^-|z'|
//
// With z' in hand, t is one ex2.approx.f16x2 whose argument's negated
// absolute value folds into the instruction, so the scaling multiply of
// softplus_f16x2 disappears: five instructions per pair.  log2(1 + t) on
// [0, 1] is the polynomial above times log2 e (exact scaling of the same
// minimax fit): 1.42459526, -0.58921265, 0.16538906, rounded to fp16
// 1.42480469, -0.58935547, 0.16540527 (max |error| 5.9e-4 in natural units).
// A chain in these units needs log2 e applied once to its first layer's
// result and ln 2 to its last (scale_pack_f16x2), and its later biases
// scaled by log2 e; the weights are unchanged, since ln 2 log2 e = 1.
constexpr uint32_t kLog2pC1X2 = 0x3DB33DB3u;
constexpr uint32_t kLog2pC2X2 = 0xB8B7B8B7u;
constexpr uint32_t kLog2pC3X2 = 0x314B314Bu;
constexpr float kLog2e = 1.44269504088896341f;
constexpr float kLn2 = 0.693147180559945309f;

__device__ __forceinline__ uint32_t softplus_log2_f16x2(uint32_t z) {
  const uint32_t c1 = kLog2pC1X2;
  const uint32_t c2 = kLog2pC2X2;
  const uint32_t c3 = kLog2pC3X2;
  uint32_t a, t, q, r, h;
  asm("abs.f16x2 %0, %1;" : "=r"(a) : "r"(z));  // |z'| and its negation fold into the ex2
  asm("neg.f16x2 %0, %1;" : "=r"(a) : "r"(a));
  asm("ex2.approx.f16x2 %0, %1;" : "=r"(t) : "r"(a));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(q) : "r"(c3), "r"(t), "r"(c2));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(q) : "r"(q), "r"(t), "r"(c1));
  asm("max.f16x2 %0, %1, %2;" : "=r"(r) : "r"(z), "r"(0u));
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(h) : "r"(q), "r"(t), "r"(r));
  return h;
}

// (lo, hi) * s in fp32 (one packed multiply), then RNE to an fp16 pair.
__device__ __forceinline__ uint32_t scale_pack_f16x2(uint32_t lo, uint32_t hi, float s) {
  const uint64_t s2 = (static_cast<uint64_t>(__float_as_uint(s)) << 32) | __float_as_uint(s);
  uint32_t h;
  asm("{\n\t.reg .b64 a, d;\n\t.reg .b32 x, y;\n\t"
      "mov.b64 a, {%1, %2};\n\t"
      "mul.rn.f32x2 d, a, %3;\n\t"
      "mov.b64 {x, y}, d;\n\t"
      "cvt.rn.f16x2.f32 %0, y, x;\n\t}"
      : "=r"(h)
      : "r"(lo), "r"(hi), "l"(s2));
  return h;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// act'(h) from the activation's output h: softplus' = sigmoid(z) = 1 - e^-h
// (e^h = 1 + e^z), ReLU' = [h > 0], identity' = 1.
template <int kAct>
__device__ __forceinline__ float dact_from_output(float h) {
  if constexpr (kAct == kActSoftplus) {
    return 1.0f - __expf(-h);  // absolute error ~1e-7: the product is rounded to 16 bits
  } else if constexpr (kAct == kActRelu) {
    return h > 0.0f ? 1.0f : 0.0f;
  } else {
    return 1.0f;
  }
}

}  // namespace coalesce
