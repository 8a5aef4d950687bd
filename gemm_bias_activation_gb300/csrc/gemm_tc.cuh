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
      const float y0 = act_apply_16<kAct>(__uint_as_float(r[8 * g + 2 * i]) + bv[2 * i]);
      const float y1 = act_apply_16<kAct>(__uint_as_float(r[8 * g + 2 * i + 1]) + bv[2 * i + 1]);
      w[i] = pack2(y0, y1, kBF16);
    }
    const uint32_t chunk = static_cast<uint32_t>(g) ^ (lane & 7u);
    *reinterpret_cast<uint4*>(buf + lane * 128u + chunk * 16u) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace tcgemm
}  // namespace coalesce
