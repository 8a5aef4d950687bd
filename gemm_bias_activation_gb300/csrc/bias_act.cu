// In-place bias + activation over a row-major [M, N] matrix:
//
//   Y[i, j] = act(Y[i, j] + bias[j])
//
// This is the second kernel of the UNFUSED sequence that the "Coalesce"
// README's "Fusion study (03_matmul_fused)" compares the fused kernel with
// (the same matmul, followed by a separate elementwise kernel).  It exists to
// measure what fusion saves and to check that both orders agree; the fused
// entry point never uses it.
//
// HBM-bound by construction: one 16-byte vector load and store per thread per
// step (8 values for fp16/bf16, 4 for fp32), grid-stride over the matrix with
// the grid a multiple of the SM count.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "epilogue.cuh"
#include "internal.h"

namespace coalesce {
namespace biasact {

template <typename T>
struct Vec;

template <>
struct Vec<float> {
  static constexpr int kN = 4;
  __device__ static void to_f32(const uint4& v, float* f) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  __device__ static uint4 from_f32(const float* f) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
  }
};

template <>
struct Vec<__half> {
  static constexpr int kN = 8;
  __device__ static void to_f32(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 p = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      f[2 * i] = p.x;
      f[2 * i + 1] = p.y;
    }
  }
  __device__ static uint4 from_f32(const float* f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

template <>
struct Vec<__nv_bfloat16> {
  static constexpr int kN = 8;
  __device__ static void to_f32(const uint4& v, float* f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
      f[2 * i] = p.x;
      f[2 * i + 1] = p.y;
    }
  }
  __device__ static uint4 from_f32(const float* f) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

template <typename T, int kAct>
__global__ void __launch_bounds__(256) bias_act_kernel(T* __restrict__ Y, const T* __restrict__ bias, int64_t M,
                                                       int64_t N) {
  constexpr int V = Vec<T>::kN;
  const int64_t vec_per_row = N / V;  // N is a multiple of V (16-byte rows)
  const int64_t total = M * vec_per_row;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t col = (idx % vec_per_row) * V;
    uint4* p = reinterpret_cast<uint4*>(Y) + idx;
    float y[V], b[V];
    Vec<T>::to_f32(*p, y);
    if (bias != nullptr) {
      Vec<T>::to_f32(__ldg(reinterpret_cast<const uint4*>(bias + col)), b);
    } else {
#pragma unroll
      for (int i = 0; i < V; ++i) b[i] = 0.0f;
    }
#pragma unroll
    for (int i = 0; i < V; ++i) y[i] = act_apply<kAct>(y[i] + b[i]);
    *p = Vec<T>::from_f32(y);
  }
}

template <typename T>
cudaError_t launch_typed(const DeviceCtx& dev, int64_t M, int64_t N, void* Y, const void* bias, int act,
                         cudaStream_t stream) {
  constexpr int V = Vec<T>::kN;
  const int64_t total = M * (N / V);
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(dev.sm_count) * 8;  // 8 CTAs of 256 threads per SM
  if (blocks > cap) blocks = cap;
  T* y = static_cast<T*>(Y);
  const T* b = static_cast<const T*>(bias);
  switch (act) {
    case kActRelu:
      bias_act_kernel<T, kActRelu><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(y, b, M, N);
      break;
    case kActGeluErf:
      bias_act_kernel<T, kActGeluErf><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(y, b, M, N);
      break;
    case kActSoftplus:
      bias_act_kernel<T, kActSoftplus><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(y, b, M, N);
      break;
    default:
      bias_act_kernel<T, kActNone><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(y, b, M, N);
      break;
  }
  return cudaGetLastError();
}

}  // namespace biasact

cudaError_t launch_bias_act(const DeviceCtx& dev, int dtype_code, int64_t M, int64_t N, void* Y, const void* bias,
                            int act, cudaStream_t stream) {
  using namespace biasact;
  switch (dtype_code) {
    case 0:
      return launch_typed<float>(dev, M, N, Y, bias, act, stream);
    case 1:
      return launch_typed<__half>(dev, M, N, Y, bias, act, stream);
    default:
      return launch_typed<__nv_bfloat16>(dev, M, N, Y, bias, act, stream);
  }
}

}  // namespace coalesce
