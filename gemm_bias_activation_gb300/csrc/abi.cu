// The C ABI of libcoalesce (declared in include/coalesce.h): argument checks,
// per-device state, TMA descriptor encoding and dispatch to the kernels.
//
// Every argument check runs before the first CUDA call, so a rejected call
// enqueues nothing and touches no output, and the checks work on a machine
// without a GPU.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "coalesce.h"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace coalesce {

// Error word written by the kernels' bounded waits (one copy per device), and
// the word coalesce_device_status moves it into (atomically, clearing it).
__device__ uint32_t g_wait_error_word;
__device__ uint32_t g_status_snapshot;

namespace {

constexpr int kMaxDevices = 64;

std::mutex g_mutex;
DeviceCtx g_devices[kMaxDevices];
bool g_device_ready[kMaxDevices] = {};

thread_local char g_last_error[256] = "no error";

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode_tiled = nullptr;

int record_cuda(cudaError_t e, const char* where) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
  return COALESCE_ERR_CUDA;
}

// Fill (once per device) the SM count and the device address of the error word.
int current_device_ctx(const DeviceCtx** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return record_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) {
    snprintf(g_last_error, sizeof(g_last_error), "device ordinal %d out of range", dev);
    return COALESCE_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_device_ready[dev]) {
    DeviceCtx c;
    c.device = dev;
    if ((e = cudaDeviceGetAttribute(&c.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return record_cuda(e, "cudaDeviceGetAttribute");
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3) {
      snprintf(g_last_error, sizeof(g_last_error), "device %d is sm_%d%d; this library is built for sm_103a", dev,
               major, minor);
      return COALESCE_ERR_UNSUPPORTED;
    }
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_wait_error_word)) != cudaSuccess)
      return record_cuda(e, "cudaGetSymbolAddress");
    c.err_word = static_cast<uint32_t*>(p);
    if ((e = cudaGetSymbolAddress(&p, g_status_snapshot)) != cudaSuccess)
      return record_cuda(e, "cudaGetSymbolAddress");
    c.status_snapshot = static_cast<uint32_t*>(p);
    if (g_encode_tiled == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
        return record_cuda(e == cudaSuccess ? cudaErrorSymbolNotFound : e, "cuTensorMapEncodeTiled lookup");
      g_encode_tiled = reinterpret_cast<EncodeTiledFn>(fn);
    }
    g_devices[dev] = c;
    g_device_ready[dev] = true;
  }
  *out = &g_devices[dev];
  return COALESCE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, uint64_t abytes, const void* b, uint64_t bbytes) {
  if (a == nullptr || b == nullptr) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + bbytes && b0 < a0 + abytes;
}

int invalid(const char* what) {
  snprintf(g_last_error, sizeof(g_last_error), "invalid argument: %s", what);
  return COALESCE_ERR_INVALID_ARG;
}

// Waits, with the same bounded wait every kernel uses, on an mbarrier that
// nothing ever arrives on; after `limit_ns` it records kErrWaitSelfTest in the
// error word and returns, leaving the context usable.
__global__ void wait_timeout_selftest_kernel(uint32_t* err, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  mbar_wait(b, 0, err, kErrWaitSelfTest, limit_ns);
  __syncthreads();
}

// Moves the error word into the snapshot word and clears it in one atomic
// exchange, so a code set by a kernel at any moment is either reported by this
// call or left for the next one, never lost.
__global__ void status_fetch_clear_kernel(uint32_t* err, uint32_t* snapshot) { *snapshot = atomicExch(err, 0u); }

// Measurement aid: independent fp32 FMA chains, no memory traffic in the
// loop.  kChains accumulators per thread keep the FMA pipe fed across its
// latency; the loop-invariant multiplier and addend are runtime values so that
// nothing folds.  One conditional store keeps the work observable.
constexpr int kFfmaChains = 16;
constexpr int kFfmaThreads = 256;
constexpr int kFfmaBlocksPerSm = 4;
constexpr int kFfmaUnroll = 8;

__global__ void __launch_bounds__(kFfmaThreads) ffma_rate_kernel(int64_t iters, float m, float c, float* sink) {
  float a[kFfmaChains];
#pragma unroll
  for (int i = 0; i < kFfmaChains; ++i) a[i] = static_cast<float>(threadIdx.x + i);
  for (int64_t it = 0; it < iters; it += kFfmaUnroll) {
#pragma unroll
    for (int u = 0; u < kFfmaUnroll; ++u) {
#pragma unroll
      for (int i = 0; i < kFfmaChains; ++i) a[i] = fmaf(a[i], m, c);
    }
  }
  float s = 0.0f;
#pragma unroll
  for (int i = 0; i < kFfmaChains; ++i) s += a[i];
  if (s == 1234.5f) *sink = s;
}

}  // namespace

cudaError_t encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t elem_bytes, const void* base,
                           uint64_t rows, uint64_t cols, uint32_t box_rows, uint32_t box_cols,
                           CUtensorMapSwizzle swizzle) {
  if (g_encode_tiled == nullptr) return cudaErrorInitializationError;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * elem_bytes};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode_tiled(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(g_last_error, sizeof(g_last_error), "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
    return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

}  // namespace coalesce

using namespace coalesce;

extern "C" int coalesce_gemm_bias_act(int64_t M, int64_t N, int64_t K, int dtype, const void* A, const void* B,
                                      const void* bias, void* Y, int act, void* stream) {
  if (M < 1 || N < 1 || K < 1) return invalid("M, N and K must be >= 1");
  if (M > 0x7FFFFFFF || N > 0x7FFFFFFF || K > 0x7FFFFFFF) {
    snprintf(g_last_error, sizeof(g_last_error), "M, N and K must be < 2^31");
    return COALESCE_ERR_UNSUPPORTED;
  }
  if (dtype != COALESCE_F32 && dtype != COALESCE_F16 && dtype != COALESCE_BF16) return invalid("unknown dtype");
  if (act < COALESCE_ACT_NONE || act > COALESCE_ACT_SOFTPLUS) return invalid("unknown activation");
  if (A == nullptr || B == nullptr || Y == nullptr) return invalid("A, B and Y must not be NULL");
  const uint64_t esz = dtype == COALESCE_F32 ? 4 : 2;
  if (!aligned16(A) || !aligned16(B) || !aligned16(Y) || (bias != nullptr && !aligned16(bias)) ||
      (static_cast<uint64_t>(K) * esz) % 16 != 0 || (static_cast<uint64_t>(N) * esz) % 16 != 0) {
    snprintf(g_last_error, sizeof(g_last_error),
             "pointers must be 16-byte aligned and K, N multiples of %d for this dtype", static_cast<int>(16 / esz));
    return COALESCE_ERR_MISALIGNED;
  }
  const uint64_t ybytes = static_cast<uint64_t>(M) * N * esz;
  if (overlaps(Y, ybytes, A, static_cast<uint64_t>(M) * K * esz) ||
      overlaps(Y, ybytes, B, static_cast<uint64_t>(K) * N * esz) || overlaps(Y, ybytes, bias, N * esz))
    return invalid("Y overlaps an input");

  const DeviceCtx* dev = nullptr;
  int st = current_device_ctx(&dev);
  if (st != COALESCE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (dtype == COALESCE_F32) {
    e = launch_gemm_f32(*dev, M, N, K, static_cast<const float*>(A), static_cast<const float*>(B),
                        static_cast<const float*>(bias), static_cast<float*>(Y), act, s);
  } else {
    e = launch_gemm_tc(*dev, dtype == COALESCE_BF16, M, N, K, A, B, bias, Y, act, s);
  }
  if (e != cudaSuccess) return record_cuda(e, "coalesce_gemm_bias_act launch");
  return COALESCE_OK;
}

extern "C" int coalesce_gemm_ex(int64_t M, int64_t N, int64_t K, int dtype, unsigned flags, const void* A,
                                const void* B, const void* bias, const void* aux, void* Y, int act, void* stream) {
  if (flags == 0 && aux == nullptr) return coalesce_gemm_bias_act(M, N, K, dtype, A, B, bias, Y, act, stream);
  if (M < 1 || N < 1 || K < 1) return invalid("M, N and K must be >= 1");
  if (flags & ~static_cast<unsigned>(COALESCE_GEMM_TRANS_A | COALESCE_GEMM_TRANS_B | COALESCE_GEMM_ACCUM_F32 |
                                     COALESCE_GEMM_DACT))
    return invalid("unknown flag");
  if ((flags & COALESCE_GEMM_ACCUM_F32) && (flags & COALESCE_GEMM_DACT))
    return invalid("ACCUM_F32 and DACT are exclusive");
  if (dtype != COALESCE_F32 && dtype != COALESCE_F16 && dtype != COALESCE_BF16) return invalid("unknown dtype");
  if (act < COALESCE_ACT_NONE || act > COALESCE_ACT_SOFTPLUS) return invalid("unknown activation");
  if (A == nullptr || B == nullptr || Y == nullptr) return invalid("A, B and Y must not be NULL");
  const bool ta = (flags & COALESCE_GEMM_TRANS_A) != 0, tb = (flags & COALESCE_GEMM_TRANS_B) != 0;
  const bool acc = (flags & COALESCE_GEMM_ACCUM_F32) != 0, dact = (flags & COALESCE_GEMM_DACT) != 0;
  if (acc && (bias != nullptr || act != COALESCE_ACT_NONE)) return invalid("ACCUM_F32 takes no bias and no activation");
  if (dact && (aux == nullptr || bias != nullptr)) return invalid("DACT needs aux and takes no bias");
  if (!dact && aux != nullptr) return invalid("aux is only read with DACT");
  if (dtype == COALESCE_F32 || (dact && act == COALESCE_ACT_GELU_ERF) || M > 0x7FFFFFFF || N > 0x7FFFFFFF ||
      K > 0x7FFFFFFF) {
    snprintf(g_last_error, sizeof(g_last_error),
             "these flags need fp16/bf16, sizes < 2^31, and (DACT) an activation whose derivative follows from "
             "its output (none, relu, softplus)");
    return COALESCE_ERR_UNSUPPORTED;
  }
  // Row strides (elements): A is [M, K] or [K, M], B is [K, N] or [N, K], Y and aux [M, N].
  const int64_t a_ld = ta ? M : K, b_ld = tb ? K : N;
  if (!aligned16(A) || !aligned16(B) || !aligned16(Y) || (aux != nullptr && !aligned16(aux)) || a_ld % 8 != 0 ||
      b_ld % 8 != 0 || N % (acc ? 4 : 8) != 0) {
    snprintf(g_last_error, sizeof(g_last_error),
             "pointers must be 16-byte aligned and every row stride a multiple of 16 bytes");
    return COALESCE_ERR_MISALIGNED;
  }
  const uint64_t ybytes = static_cast<uint64_t>(M) * N * (acc ? 4 : 2);
  if (overlaps(Y, ybytes, A, static_cast<uint64_t>(M) * K * 2) ||
      overlaps(Y, ybytes, B, static_cast<uint64_t>(K) * N * 2))
    return invalid("Y overlaps an input");
  // aux may be Y itself (each element is read before the store that covers it), but not partly.
  if (aux != nullptr && aux != Y && overlaps(Y, ybytes, aux, static_cast<uint64_t>(M) * N * 2))
    return invalid("aux partly overlaps Y");

  const DeviceCtx* dev = nullptr;
  int st = current_device_ctx(&dev);
  if (st != COALESCE_OK) return st;
  cudaError_t e = launch_gemm_tc_ex(*dev, dtype == COALESCE_BF16, ta, tb, acc ? 1 : dact ? 2 : 0, M, N, K, A, B, bias,
                                    aux, Y, act, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return record_cuda(e, "coalesce_gemm_ex launch");
  return COALESCE_OK;
}

extern "C" int coalesce_bias_act(int64_t M, int64_t N, int dtype, void* Y, const void* bias, int act,
                                 void* stream) {
  if (M < 1 || N < 1) return invalid("M and N must be >= 1");
  if (dtype != COALESCE_F32 && dtype != COALESCE_F16 && dtype != COALESCE_BF16) return invalid("unknown dtype");
  if (act < COALESCE_ACT_NONE || act > COALESCE_ACT_SOFTPLUS) return invalid("unknown activation");
  if (Y == nullptr) return invalid("Y must not be NULL");
  const uint64_t esz = dtype == COALESCE_F32 ? 4 : 2;
  if (!aligned16(Y) || (bias != nullptr && !aligned16(bias)) || (static_cast<uint64_t>(N) * esz) % 16 != 0) {
    snprintf(g_last_error, sizeof(g_last_error), "pointers must be 16-byte aligned and N a multiple of %d",
             static_cast<int>(16 / esz));
    return COALESCE_ERR_MISALIGNED;
  }
  if (overlaps(Y, static_cast<uint64_t>(M) * N * esz, bias, N * esz)) return invalid("Y overlaps bias");
  const DeviceCtx* dev = nullptr;
  int st = current_device_ctx(&dev);
  if (st != COALESCE_OK) return st;
  cudaError_t e = launch_bias_act(*dev, dtype, M, N, Y, bias, act, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return record_cuda(e, "coalesce_bias_act launch");
  return COALESCE_OK;
}

extern "C" int coalesce_mlp_fused_ex(int64_t rows, int64_t D, int64_t H, int64_t O, int L, int dtype, const void* x,
                                     const void* const* W, const void* const* b, void* out, int act,
                                     void* stream) {
  if (rows < 1 || D < 1 || H < 1 || O < 1 || L < 1) return invalid("rows, D, H, O and L must be >= 1");
  if (dtype < COALESCE_F32 || dtype > COALESCE_BF16) return invalid("unknown dtype");
  if (act < COALESCE_ACT_NONE || act > COALESCE_ACT_SOFTPLUS) return invalid("unknown activation");
  if (x == nullptr || W == nullptr || out == nullptr) return invalid("x, W and out must not be NULL");
  if (dtype == COALESCE_F32) {
    snprintf(g_last_error, sizeof(g_last_error), "the chained MLP runs on the tensor cores: fp16 or bf16 only");
    return COALESCE_ERR_UNSUPPORTED;
  }
  if (L > 8) {
    snprintf(g_last_error, sizeof(g_last_error), "at most 8 layers");
    return COALESCE_ERR_UNSUPPORTED;
  }
  for (int l = 0; l < L; ++l)
    if (W[l] == nullptr) return invalid("W[l] must not be NULL");
  if (D > 256 || H > 256 || O > 256 || rows > 0x7FFFFFFF) {
    snprintf(g_last_error, sizeof(g_last_error), "D, H and O must be at most 256, L <= 8 and rows < 2^31");
    return COALESCE_ERR_UNSUPPORTED;
  }
  if (D % 8 != 0 || H % 8 != 0 || O % 8 != 0) {
    snprintf(g_last_error, sizeof(g_last_error), "D, H and O must be multiples of 8 (16-byte rows)");
    return COALESCE_ERR_MISALIGNED;
  }
  bool al = aligned16(x) && aligned16(out);
  for (int l = 0; l < L; ++l) {
    al = al && aligned16(W[l]);
    if (b != nullptr && b[l] != nullptr) al = al && aligned16(b[l]);
  }
  if (!al) {
    snprintf(g_last_error, sizeof(g_last_error), "pointers must be 16-byte aligned");
    return COALESCE_ERR_MISALIGNED;
  }
  const uint64_t obytes = static_cast<uint64_t>(rows) * O * 2;
  if (overlaps(out, obytes, x, static_cast<uint64_t>(rows) * D * 2)) return invalid("out overlaps x");

  const DeviceCtx* dev = nullptr;
  int st = current_device_ctx(&dev);
  if (st != COALESCE_OK) return st;
  cudaError_t e = launch_mlp_fused(*dev, rows, static_cast<int>(D), static_cast<int>(H), static_cast<int>(O), L,
                                   dtype == COALESCE_BF16, x, W, b, out, act, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) {
    snprintf(g_last_error, sizeof(g_last_error), "this MLP shape is not implemented");
    return COALESCE_ERR_UNSUPPORTED;
  }
  if (e != cudaSuccess) return record_cuda(e, "coalesce_mlp_fused launch");
  return COALESCE_OK;
}

extern "C" int coalesce_mlp_fused(int64_t rows, int64_t D, int64_t H, int L, const void* x, const void* const* W,
                                  const void* const* b, void* out, int act, void* stream) {
  return coalesce_mlp_fused_ex(rows, D, H, H, L, COALESCE_F16, x, W, b, out, act, stream);
}

namespace {

// Common checks of the training entry points; fills `wbytes` per layer.
int check_train_shapes(int64_t rows, int64_t D, int64_t H, int64_t O, int L, int dtype, int act) {
  if (rows < 1 || D < 1 || H < 1 || O < 1 || L < 1) return invalid("rows, D, H, O and L must be >= 1");
  if (dtype != COALESCE_F32 && dtype != COALESCE_F16 && dtype != COALESCE_BF16) return invalid("unknown dtype");
  if (act < COALESCE_ACT_NONE || act > COALESCE_ACT_SOFTPLUS) return invalid("unknown activation");
  if (dtype == COALESCE_F32 || act == COALESCE_ACT_GELU_ERF || L > 8 || rows > 0x7FFFFFFF || D > 0x7FFFFFFF ||
      H > 0x7FFFFFFF || O > 0x7FFFFFFF) {
    snprintf(g_last_error, sizeof(g_last_error),
             "training needs fp16/bf16, L <= 8, sizes < 2^31 and an activation whose derivative follows from its "
             "output (none, relu, softplus)");
    return COALESCE_ERR_UNSUPPORTED;
  }
  if (D % 8 != 0 || H % 8 != 0 || O % 8 != 0) {
    snprintf(g_last_error, sizeof(g_last_error), "D, H and O must be multiples of 8 (16-byte rows)");
    return COALESCE_ERR_MISALIGNED;
  }
  return COALESCE_OK;
}

}  // namespace

extern "C" int coalesce_mlp_forward_train(int64_t rows, int64_t D, int64_t H, int64_t O, int L, int dtype,
                                          const void* x, const void* const* W, const void* const* b, void* const* h,
                                          void* out, int act, void* stream) {
  int st = check_train_shapes(rows, D, H, O, L, dtype, act);
  if (st != COALESCE_OK) return st;
  if (x == nullptr || W == nullptr || out == nullptr || (L > 1 && h == nullptr))
    return invalid("x, W, h and out must not be NULL");
  bool al = aligned16(x) && aligned16(out);
  for (int l = 0; l < L; ++l) {
    if (W[l] == nullptr || (l < L - 1 && h[l] == nullptr)) return invalid("W[l] and h[l] must not be NULL");
    al = al && aligned16(W[l]) && (l == L - 1 || aligned16(h[l])) &&
         (b == nullptr || b[l] == nullptr || aligned16(b[l]));
  }
  if (!al) {
    snprintf(g_last_error, sizeof(g_last_error), "pointers must be 16-byte aligned");
    return COALESCE_ERR_MISALIGNED;
  }
  const DeviceCtx* dev = nullptr;
  if ((st = current_device_ctx(&dev)) != COALESCE_OK) return st;
  cudaError_t e = launch_mlp_forward_train(*dev, rows, D, H, O, L, dtype == COALESCE_BF16, x, W, b, h, out, act,
                                           static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return record_cuda(e, "coalesce_mlp_forward_train launch");
  return COALESCE_OK;
}

extern "C" int coalesce_mlp_backward(int64_t rows, int64_t D, int64_t H, int64_t O, int L, int dtype, const void* x,
                                     const void* const* W, void* const* h, const void* dout, void* dx,
                                     float* const* dW, float* const* db, int act, void* stream) {
  int st = check_train_shapes(rows, D, H, O, L, dtype, act);
  if (st != COALESCE_OK) return st;
  if (x == nullptr || W == nullptr || dout == nullptr || dW == nullptr || (L > 1 && h == nullptr))
    return invalid("x, W, h, dout and dW must not be NULL");
  bool al = aligned16(x) && aligned16(dout) && (dx == nullptr || aligned16(dx));
  for (int l = 0; l < L; ++l) {
    if (W[l] == nullptr || dW[l] == nullptr || (l < L - 1 && h[l] == nullptr))
      return invalid("W[l], dW[l] and h[l] must not be NULL");
    al = al && aligned16(W[l]) && aligned16(dW[l]) && (l == L - 1 || aligned16(h[l])) &&
         (db == nullptr || db[l] == nullptr || aligned16(db[l]));
  }
  if (!al) {
    snprintf(g_last_error, sizeof(g_last_error), "pointers must be 16-byte aligned");
    return COALESCE_ERR_MISALIGNED;
  }
  if (dx != nullptr && overlaps(dx, static_cast<uint64_t>(rows) * D * 2, x, static_cast<uint64_t>(rows) * D * 2))
    return invalid("dx overlaps x");
  const DeviceCtx* dev = nullptr;
  if ((st = current_device_ctx(&dev)) != COALESCE_OK) return st;
  cudaError_t e = launch_mlp_backward(*dev, rows, D, H, O, L, dtype == COALESCE_BF16, x, W, h, dout, dx, dW, db, act,
                                      static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return record_cuda(e, "coalesce_mlp_backward launch");
  return COALESCE_OK;
}

extern "C" int coalesce_device_status(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return record_cuda(e, "cudaStreamSynchronize");
  const DeviceCtx* dev = nullptr;
  int st = current_device_ctx(&dev);
  if (st != COALESCE_OK) return st;
  status_fetch_clear_kernel<<<1, 1, 0, s>>>(dev->err_word, dev->status_snapshot);
  if ((e = cudaGetLastError()) != cudaSuccess) return record_cuda(e, "status exchange launch");
  uint32_t word = 0;
  if ((e = cudaMemcpyAsync(&word, dev->status_snapshot, sizeof(word), cudaMemcpyDeviceToHost, s)) != cudaSuccess)
    return record_cuda(e, "cudaMemcpyAsync(error word)");
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return record_cuda(e, "cudaStreamSynchronize");
  if (word != 0) {
    snprintf(g_last_error, sizeof(g_last_error), "a kernel's bounded wait ran out (error word 0x%x)", word);
    return COALESCE_ERR_DEVICE_TIMEOUT;
  }
  return COALESCE_OK;
}

extern "C" int coalesce_measure_ffma(int64_t iters, float* sink, double* flop, void* stream) {
  if (iters < kFfmaUnroll || iters > (int64_t{1} << 40) || iters % kFfmaUnroll != 0)
    return invalid("iters must be a positive multiple of 8, at most 2^40");
  if (sink == nullptr || flop == nullptr) return invalid("sink and flop must not be NULL");
  const DeviceCtx* dev = nullptr;
  int st = current_device_ctx(&dev);
  if (st != COALESCE_OK) return st;
  const int blocks = dev->sm_count * kFfmaBlocksPerSm;
  // m = 1 - 2^-20 and c = 2^-20 keep every chain bounded and normal.
  ffma_rate_kernel<<<blocks, kFfmaThreads, 0, static_cast<cudaStream_t>(stream)>>>(iters, 1.0f - 0x1p-20f, 0x1p-20f,
                                                                                    sink);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return record_cuda(e, "coalesce_measure_ffma launch");
  *flop = 2.0 * static_cast<double>(blocks) * kFfmaThreads * kFfmaChains * static_cast<double>(iters);
  return COALESCE_OK;
}

extern "C" int coalesce_selftest_wait_timeout(uint64_t limit_ns, void* stream) {
  if (limit_ns < 1000 || limit_ns > 10000000000ull) return invalid("limit_ns must be in [1 us, 10 s]");
  const DeviceCtx* dev = nullptr;
  int st = current_device_ctx(&dev);
  if (st != COALESCE_OK) return st;
  wait_timeout_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev->err_word, limit_ns);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return record_cuda(e, "coalesce_selftest_wait_timeout launch");
  return COALESCE_OK;
}

extern "C" const char* coalesce_status_string(int status) {
  switch (status) {
    case COALESCE_OK:
      return "ok";
    case COALESCE_ERR_INVALID_ARG:
      return "invalid argument";
    case COALESCE_ERR_UNSUPPORTED:
      return "unsupported";
    case COALESCE_ERR_MISALIGNED:
      return "misaligned pointer or row stride";
    case COALESCE_ERR_CUDA:
      return "CUDA error";
    case COALESCE_ERR_DEVICE_TIMEOUT:
      return "device wait timed out";
    default:
      return "unknown status";
  }
}

extern "C" const char* coalesce_last_error(void) { return g_last_error; }

extern "C" void coalesce_shutdown(void) {
  std::lock_guard<std::mutex> lock(g_mutex);
  for (int i = 0; i < kMaxDevices; ++i) g_device_ready[i] = false;
}
