// Shared pieces of the tcgen05 GEMM kernels: tile shape, shared-memory
// layout, tile order and the epilogue helpers.  gemm_tc.cu holds the forward
// GEMM with bias + activation, gemm_tc_ex.cu its general form for the MLP
// backward; each kernel lives in its own translation unit.
#pragma once

#include "epilogue.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace coalesce {
namespace tcgemm {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int kEpiWarps = 4;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kGroupM = 32;

constexpr uint32_t kABytes = BM * BK * 2;        // 16 KiB
constexpr uint32_t kBChunkBytes = BK * 64 * 2;   // 8 KiB: 64 k-rows x 64 n (128 B)
constexpr uint32_t kBBytes = BK * BN * 2;        // 32 KiB
constexpr uint32_t kOutBufBytes = 32 * 64 * 2;   // 32 rows x 64 cols
constexpr uint32_t kTmemCols = 2 * BN;

constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffB = kOffA + STAGES * kABytes;
constexpr uint32_t kOffOut = kOffB + STAGES * kBBytes;
constexpr uint32_t kOffBars = kOffOut + kEpiWarps * 2 * kOutBufBytes;
constexpr uint32_t kNumBars = 2 * STAGES + 4 + 1;  // full, empty, acc_full x2, acc_empty x2, mma_done
constexpr uint32_t kOffTmemSlot = kOffBars + kNumBars * 8;
constexpr uint32_t kSmemBytes = kOffTmemSlot + 16 + 1024;  // + slack to align the base to 1 KiB

static_assert(kSmemBytes <= 232448, "shared memory budget exceeded");

__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, int& mb, int& nb) {
  const int per_group = kGroupM * num_n;
  const int group = t / per_group;
  const int first_m = group * kGroupM;
  const int gm = min(num_m - first_m, kGroupM);
  const int r = t - group * per_group;
  mb = first_m + r % gm;
  nb = r / gm;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi, bool bf16) {
  if (bf16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

__device__ __forceinline__ void unpack8(uint4 v, bool bf16, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (bf16) {
      __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
      float2 p = __bfloat1622float2(h);
      f[2 * i] = p.x;
      f[2 * i + 1] = p.y;
    } else {
      __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
      float2 p = __half22float2(h);
      f[2 * i] = p.x;
      f[2 * i + 1] = p.y;
    }
  }
}

// Packed fp32 pair arithmetic (one add.rn.f32x2 / mul.rn.f32x2 per pair):
// the same roundings as two scalar operations.
__device__ __forceinline__ float2 f2_add(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 x, y, d;\n\t"
      "mov.b64 x, {%2, %3};\n\t"
      "mov.b64 y, {%4, %5};\n\t"
      "add.rn.f32x2 d, x, y;\n\t"
      "mov.b64 {%0, %1}, d;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

__device__ __forceinline__ float2 f2_mul(float2 a, float2 b) {
  float2 r;
  asm("{\n\t.reg .b64 x, y, d;\n\t"
      "mov.b64 x, {%2, %3};\n\t"
      "mov.b64 y, {%4, %5};\n\t"
      "mul.rn.f32x2 d, x, y;\n\t"
      "mov.b64 {%0, %1}, d;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}

// The activation on a pair of fp32 values z (bias already added).  GELU
// keeps its scalar form's operations and order, 0.5 z (1 + erf(z / sqrt 2)),
// with everything but erff on packed pairs; the others go value by value.
template <int kAct>
__device__ __forceinline__ float2 act_pair_f32(float2 z) {
  if constexpr (kAct == kActGeluErf) {
    const float2 u = f2_mul(z, make_float2(0.70710678118654752f, 0.70710678118654752f));
    const float2 t = f2_add(make_float2(1.0f, 1.0f), make_float2(erff(u.x), erff(u.y)));
    return f2_mul(f2_mul(make_float2(0.5f, 0.5f), z), t);
  } else {
    return make_float2(act_apply_16<kAct>(z.x), act_apply_16<kAct>(z.y));
  }
}

// One 32-row x 64-column slice: bias + activation + downcast, written row
// `lane` of the 128-B-swizzled staging buffer (16-B chunk j of row r lives at
// chunk j ^ (r & 7), the layout a SWIZZLE_128B TMA store expects).
template <bool kBF16, int kAct>
__device__ __forceinline__ void epilogue_slice(const uint32_t* r, const uint16_t* __restrict__ bias, int n0, int N,
                                               uint8_t* buf, uint32_t lane) {
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    float bv[8];
    const int nc = n0 + 8 * g;
    if (bias != nullptr && nc < N) {
      // N is a multiple of 8, so a group of 8 columns is entirely inside or outside.
      unpack8(__ldg(reinterpret_cast<const uint4*>(bias + nc)), kBF16, bv);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) bv[i] = 0.0f;
    }
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 z = f2_add(make_float2(__uint_as_float(r[8 * g + 2 * i]), __uint_as_float(r[8 * g + 2 * i + 1])),
                              make_float2(bv[2 * i], bv[2 * i + 1]));
      const float2 y = act_pair_f32<kAct>(z);
      w[i] = pack2(y.x, y.y, kBF16);
    }
    const uint32_t chunk = static_cast<uint32_t>(g) ^ (lane & 7u);
    *reinterpret_cast<uint4*>(buf + lane * 128u + chunk * 16u) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace tcgemm
}  // namespace coalesce
