// Training side of the chained MLP: the forward pass that keeps every layer's
// activation, and the backward pass (data and parameter gradients).
//
// The "MLP Megakernel" README ("Key ideas") trains the chain with a fused
// backward for small batches and, above 32K rows, with GEMMs for the weight
// gradients interleaved with the data-gradient computation.  The workloads
// here have 2^20..2^22 rows, so this file is the GEMM form, on the library's
// own tcgen05 GEMM (gemm_tc.cu):
//
//   forward   h_0 = x, h_l = act(h_{l-1} W_l + b_l) stored for l < L,
//             out = h_{L-1} W_L + b_L                 (the fused chain, which
//                                                     stores the h_l on its
//                                                     way, or L GEMM calls)
//   backward  g_L = dout; for l = L .. 1:
//               db_l = sum over rows of g_l            (column-sum kernel)
//               dW_l = h_{l-1}^T g_l                   (fp32, K = rows split
//                                                       over all SMs)
//               g_{l-1} = (g_l W_l^T) * act'(h_{l-1})  (l > 1; in place over
//                                                       h_{l-1}, which no
//                                                       later step reads)
//               dx = g_1 W_1^T                         (l = 1)
//
// act' comes from the stored activation itself: softplus' = sigmoid(z) =
// 1 - e^-h (e^h = 1 + e^z), ReLU' = [h > 0].  The README keeps fp32
// activations for this derivative; here they are stored in the operand type
// (fp16/bf16), which the next GEMM consumes anyway, and the derivative is
// evaluated in fp32 from them.  No device memory is allocated: the data
// gradients overwrite the stored activations.
#include "internal.h"
#include "epilogue.cuh"

#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace coalesce {
namespace train {

constexpr int kColThreads = 256;
constexpr int kColRows = 2048;  // rows per block

// db[n] += sum over this block's rows of g[r][n], g [rows, N] 16-bit
// row-major; a warp covers 64 columns (a column pair per lane, 128 B per row
// read), eight warps split the rows, the block reduces in shared memory and
// adds into db (fp32, zeroed by the caller) with one atomic per column.
template <bool kBF16>
__global__ void __launch_bounds__(kColThreads)
    colsum_kernel(const uint16_t* __restrict__ g, float* __restrict__ db, int rows, int N) {
  __shared__ float part[kColThreads / 32][64];
  const int lane = threadIdx.x % 32;
  const int wy = threadIdx.x / 32;
  const int c = blockIdx.x * 64 + 2 * lane;  // N % 8 == 0: a pair is inside or outside
  const int r0 = blockIdx.y * kColRows;
  const int r1 = min(rows, r0 + kColRows);
  float s0 = 0.0f, s1 = 0.0f;
  if (c < N) {
    for (int r = r0 + wy; r < r1; r += kColThreads / 32) {
      const uint32_t bits = __ldg(reinterpret_cast<const unsigned int*>(g + static_cast<size_t>(r) * N + c));
      float2 v;
      if (kBF16) {
        v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bits));
      } else {
        v = __half22float2(*reinterpret_cast<const __half2*>(&bits));
      }
      s0 += v.x;
      s1 += v.y;
    }
  }
  part[wy][2 * lane] = s0;
  part[wy][2 * lane + 1] = s1;
  __syncthreads();
  if (threadIdx.x < 64) {
    float t = 0.0f;
#pragma unroll
    for (int w = 0; w < kColThreads / 32; ++w) t += part[w][threadIdx.x];
    const int col = blockIdx.x * 64 + static_cast<int>(threadIdx.x);
    if (col < N) atomicAdd(db + col, t);
  }
}

}  // namespace train

// Width of layer l's output in an L-layer chain D -> H -> ... -> H -> O.
static inline int64_t out_width(int64_t H, int64_t O, int L, int l) { return l == L - 1 ? O : H; }
static inline int64_t in_width(int64_t D, int64_t H, int l) { return l == 0 ? D : H; }

cudaError_t launch_mlp_forward_train(const DeviceCtx& dev, int64_t rows, int64_t D, int64_t H, int64_t O, int L,
                                     bool bf16, const void* x, const void* const* W, const void* const* b,
                                     void* const* h, void* out, int act, cudaStream_t stream) {
  // The fused chain (mlp_fused.cu) stores the activations on its way when the
  // shapes are ones it implements; other shapes go layer by layer.
  const bool fits = D <= 256 && H <= 256 && O <= 256;
  if (fits) {
    const cudaError_t e = launch_mlp_fused(dev, rows, static_cast<int>(D), static_cast<int>(H), static_cast<int>(O),
                                           L, bf16, x, W, b, out, act, stream, h);
    if (e != cudaErrorNotSupported) return e;
  }
  for (int l = 0; l < L; ++l) {
    const void* in = l == 0 ? x : h[l - 1];
    void* y = l == L - 1 ? out : h[l];
    const cudaError_t e =
        launch_gemm_tc_ex(dev, bf16, false, false, 0, rows, out_width(H, O, L, l), in_width(D, H, l), in, W[l],
                          b != nullptr ? b[l] : nullptr, nullptr, y, l == L - 1 ? kActNone : act, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_mlp_backward(const DeviceCtx& dev, int64_t rows, int64_t D, int64_t H, int64_t O, int L,
                                bool bf16, const void* x, const void* const* W, void* const* h, const void* dout,
                                void* dx, float* const* dW, float* const* db, int act, cudaStream_t stream) {
  // The fused backward where it implements the shapes; the GEMM form below
  // otherwise.
  if (mlp_backward_fused_supported(D, H, O, L)) {
    const cudaError_t e = launch_mlp_backward_fused(dev, rows, static_cast<int>(D), static_cast<int>(H),
                                                    static_cast<int>(O), L, bf16, x, W, h, dout, dx, dW, db, act,
                                                    stream);
    if (e != cudaErrorNotSupported) return e;
  }
  cudaError_t e;
  for (int l = L - 1; l >= 0; --l) {
    const int64_t K_l = in_width(D, H, l), N_l = out_width(H, O, L, l);
    const void* g = l == L - 1 ? dout : h[l];    // gradient w.r.t. this layer's pre-activation
    const void* hin = l == 0 ? x : h[l - 1];     // this layer's input
    if (db != nullptr && db[l] != nullptr) {
      if ((e = cudaMemsetAsync(db[l], 0, sizeof(float) * N_l, stream)) != cudaSuccess) return e;
      const dim3 grid(static_cast<unsigned>((N_l + 63) / 64),
                      static_cast<unsigned>((rows + train::kColRows - 1) / train::kColRows));
      if (bf16) {
        train::colsum_kernel<true><<<grid, train::kColThreads, 0, stream>>>(
            static_cast<const uint16_t*>(g), db[l], static_cast<int>(rows), static_cast<int>(N_l));
      } else {
        train::colsum_kernel<false><<<grid, train::kColThreads, 0, stream>>>(
            static_cast<const uint16_t*>(g), db[l], static_cast<int>(rows), static_cast<int>(N_l));
      }
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // dW_l = hin^T g: M = K_l, N = N_l, K = rows; hin is [rows, K_l] = At.
    if ((e = cudaMemsetAsync(dW[l], 0, sizeof(float) * K_l * N_l, stream)) != cudaSuccess) return e;
    if ((e = launch_gemm_tc_ex(dev, bf16, true, false, 1, K_l, N_l, rows, hin, g, nullptr, nullptr, dW[l], kActNone,
                               stream)) != cudaSuccess)
      return e;
    // g W_l^T: M = rows, N = K_l, K = N_l; W_l is [K_l, N_l] = Bt.
    if (l > 0) {
      // through the activation, in place over h[l-1] (its last reader was dW_l above)
      if ((e = launch_gemm_tc_ex(dev, bf16, false, true, 2, rows, K_l, N_l, g, W[l], nullptr, h[l - 1], h[l - 1], act,
                                 stream)) != cudaSuccess)
        return e;
    } else if (dx != nullptr) {
      if ((e = launch_gemm_tc_ex(dev, bf16, false, true, 0, rows, K_l, N_l, g, W[l], nullptr, nullptr, dx, kActNone,
                                 stream)) != cudaSuccess)
        return e;
    }
  }
  return cudaSuccess;
}

}  // namespace coalesce
