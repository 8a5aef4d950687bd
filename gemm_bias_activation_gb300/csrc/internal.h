// Host-side interfaces between the C ABI layer (abi.cu) and the kernel
// translation units.  Internal: nothing here is exported.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace coalesce {

// Per-device facts the launchers need, filled once per device by abi.cu.
struct DeviceCtx {
  int device = -1;
  int sm_count = 0;
  uint32_t* err_word = nullptr;  // device address of the bounded-wait error word
  uint32_t* status_snapshot = nullptr;  // device address of the word coalesce_device_status reads
};

// Encode a 2-D tiled TMA descriptor for a row-major [rows, cols] matrix of
// `elem_bytes`-sized elements (row stride = cols * elem_bytes) with a
// box of box_rows x box_cols elements and the given swizzle.  Returns
// cudaErrorInvalidValue if the driver rejects the descriptor.
cudaError_t encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t elem_bytes, const void* base,
                           uint64_t rows, uint64_t cols, uint32_t box_rows, uint32_t box_cols,
                           CUtensorMapSwizzle swizzle);

// fp16 / bf16 GEMM + bias + activation on the tcgen05 tensor cores.
cudaError_t launch_gemm_tc(const DeviceCtx& dev, bool bf16, int64_t M, int64_t N, int64_t K, const void* A,
                           const void* B, const void* bias, void* Y, int act, cudaStream_t stream);

// The same GEMM on CTA pairs (256 x 256 tiles, tcgen05 cta_group::2).
bool gemm_tc_pair_supported(int64_t M, int64_t N, int64_t K);
cudaError_t launch_gemm_tc_pair(const DeviceCtx& dev, bool bf16, int64_t M, int64_t N, int64_t K, const void* A,
                                const void* B, const void* bias, void* Y, int act, cudaStream_t stream);

// The general form used by the MLP backward.  trans_a: A given as [K, M];
// trans_b: B given as [N, K]; mode 0: Y (16-bit) = act(A B + bias); mode 1:
// Y (fp32) += A B (K split over CTAs, TMA reduce-add); mode 2: Y (16-bit) =
// (A B) * act'(aux), aux [M, N] the activation's output.
cudaError_t launch_gemm_tc_ex(const DeviceCtx& dev, bool bf16, bool trans_a, bool trans_b, int mode, int64_t M,
                              int64_t N, int64_t K, const void* A, const void* B, const void* bias, const void* aux,
                              void* Y, int act, cudaStream_t stream);

// Training side of the chained MLP (mlp_train.cu).  h: L-1 activation
// buffers [rows, H]; the backward overwrites them with data gradients.
cudaError_t launch_mlp_forward_train(const DeviceCtx& dev, int64_t rows, int64_t D, int64_t H, int64_t O, int L,
                                     bool bf16, const void* x, const void* const* W, const void* const* b,
                                     void* const* h, void* out, int act, cudaStream_t stream);
cudaError_t launch_mlp_backward(const DeviceCtx& dev, int64_t rows, int64_t D, int64_t H, int64_t O, int L,
                                bool bf16, const void* x, const void* const* W, void* const* h, const void* dout,
                                void* dx, float* const* dW, float* const* db, int act, cudaStream_t stream);

// The backward of the chained MLP as one fused kernel (mlp_backward.cu), for
// the shapes it implements (mlp_backward_fused_supported); dW and db are
// zeroed and accumulated, h is only read.
bool mlp_backward_fused_supported(int64_t D, int64_t H, int64_t O, int L);
cudaError_t launch_mlp_backward_fused(const DeviceCtx& dev, int64_t rows, int D, int H, int O, int L, bool bf16,
                                      const void* x, const void* const* W, const void* const* h, const void* dout,
                                      void* dx, float* const* dW, float* const* db, int act, cudaStream_t stream);

// fp32 GEMM + bias + activation on the FFMA pipe.
cudaError_t launch_gemm_f32(const DeviceCtx& dev, int64_t M, int64_t N, int64_t K, const float* A, const float* B,
                            const float* bias, float* Y, int act, cudaStream_t stream);

// Chained MLP (fp16 or bf16), output width O.  `W` and `b` are host arrays of
// L device pointers.
// With h != nullptr (L - 1 device pointers, [rows, H] each) every
// intermediate activation is stored as well (the training forward).
cudaError_t launch_mlp_fused(const DeviceCtx& dev, int64_t rows, int D, int H, int O, int L, bool bf16,
                             const void* x, const void* const* W, const void* const* b, void* out, int act,
                             cudaStream_t stream, void* const* h = nullptr);

// In-place Y = act(Y + bias) over a row-major [M, N] matrix (the unfused
// second pass); dtype_code is a coalesce_dtype.
cudaError_t launch_bias_act(const DeviceCtx& dev, int dtype_code, int64_t M, int64_t N, void* Y, const void* bias,
                            int act, cudaStream_t stream);


}  // namespace coalesce
