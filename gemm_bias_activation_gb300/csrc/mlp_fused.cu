// Chained MLP in one persistent kernel on the tcgen05 tensor cores (sm_103a).
//
//   h_0 = x,  h_l = act(h_{l-1} . W_l + b_l) for l < L,  out = h_{L-1} . W_L + b_L
//
// The chained MLP of the "MLP Megakernel" README ("Architecture": 3- and
// 5-layer softplus MLPs; "Key ideas": all GEMMs and activations in one
// kernel, intermediates never reach global memory, a persistent kernel that
// walks row tiles round-robin, fp16 tensor-core operands with fp32
// accumulation and conversion to fp16 only at tile boundaries).
//
// Design (one CTA per SM):
//   * All L weight matrices stay resident in shared memory for the whole
//     launch (loaded once by TMA in the MN-major, 128-B-swizzled layout the
//     MMA reads); biases are kept as fp32.
//   * E "row-tile workers" (warpgroups of 4 warps) each own H columns of
//     TMEM and two shared-memory slots of 128 rows x max(D, H) fp16.  A worker
//     runs its row tile through every layer: its leader thread issues the
//     layer's MMAs (M = 128, N = H, K = 16 steps) from the slot into TMEM;
//     the four warps read the accumulator back (tcgen05.ld, one TMEM lane =
//     one row), add the bias, apply the activation in fp32, round to fp16 and
//     write the result over the same slot in the K-major swizzled layout the
//     next layer's MMA reads.  The last layer's fp16 result is TMA-stored
//     from the slot.  Between layers nothing leaves the SM.
//   * Warp 0 is the TMA producer: it loads each worker's next x tile into the
//     worker's other slot while the worker is busy, so HBM reads, tensor-core
//     work, epilogue math and HBM writes of different tiles overlap.
// Ragged row tails are handled by TMA (zero-filled loads, clipped stores).
#include "epilogue.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace coalesce {
namespace mlp {

constexpr int BM = 128;
constexpr int kMaxLayers = 8;
constexpr int kMaxWorkers = 4;
constexpr uint32_t kSmemLimit = 232448;  // opt-in maximum dynamic shared memory per block on sm_103a
constexpr uint32_t kWeightBudget = 160u * 1024u;

struct Params {
  CUtensorMap x_map;                  // x [rows, D], box 128 x 64, 128-B swizzle
  CUtensorMap out_map;                // out [rows, H], box 32 x 64, 128-B swizzle
  CUtensorMap w_map[kMaxLayers];      // W_l [K_l, H], box K_l x 64, 128-B swizzle
  const uint16_t* bias[kMaxLayers];   // b_l[H] fp16, or nullptr
  int rows, D, H, L, act, workers;
  uint32_t* err;
};

// Shared-memory plan, identical on host and device.  Small items (barriers,
// TMEM address, fp32 biases) sit at the start of the dynamic window; the
// swizzled operand buffers start at the next 1 KiB boundary after them.
struct Layout {
  // relative to the start of dynamic shared memory
  uint32_t bar_off;        // w_full, x_full[E][2], slot_free[E][2], mma_done[E]
  uint32_t tmem_slot_off;
  uint32_t bias_off;
  uint32_t small_bytes;
  // relative to the 1 KiB-aligned big base
  uint32_t w_off[kMaxLayers];
  uint32_t slot_off;       // slot (g, s) at slot_off + (2 g + s) * slot_bytes
  uint32_t slot_bytes;
  uint32_t big_bytes;
  uint32_t alloc_bytes;    // small + worst-case alignment padding + big
  uint32_t tmem_cols;      // allocated TMEM columns (power of two)
};

__host__ __device__ inline uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

__host__ __device__ inline Layout make_layout(int D, int H, int L, int E) {
  Layout lo{};
  uint32_t off = 0;
  lo.bar_off = off;
  off += 8u * (1u + 5u * static_cast<uint32_t>(E));
  lo.tmem_slot_off = off;
  off += 16;
  lo.bias_off = off;
  off += static_cast<uint32_t>(L * H) * 4u;
  lo.small_bytes = off;
  uint32_t big = 0;
  for (int l = 0; l < L; ++l) {
    const uint32_t K = l == 0 ? D : H;
    lo.w_off[l] = big;
    big += static_cast<uint32_t>(H / 64) * K * 128u;
  }
  const int kmax = D > H ? D : H;
  lo.slot_bytes = static_cast<uint32_t>(kmax / 64) * BM * 128u;
  lo.slot_off = big;
  big += 2u * static_cast<uint32_t>(E) * lo.slot_bytes;
  lo.big_bytes = big;
  // dynamic shared memory is at least 16-byte aligned: at most 1008 bytes of padding
  lo.alloc_bytes = lo.small_bytes + 1008u + big;
  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>(E * H)) cols <<= 1;
  lo.tmem_cols = cols;
  return lo;
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// z (32 fp32 columns c0..c0+31 of this thread's row) -> + bias -> act -> fp16,
// written to row `row` of the K-major 128-B-swizzled slot (column block c0/64).
template <int kAct>
__device__ __forceinline__ void epilogue_cols32(const uint32_t* r, const float* bias_s, int c0, uint8_t* slot,
                                                uint32_t row) {
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float2 b = *reinterpret_cast<const float2*>(bias_s + c0 + 2 * i);
    const float y0 = act_apply<kAct>(__uint_as_float(r[2 * i]) + b.x);
    const float y1 = act_apply<kAct>(__uint_as_float(r[2 * i + 1]) + b.y);
    __half2 h = __floats2half2_rn(y0, y1);
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  uint8_t* rowp = slot + static_cast<uint32_t>(c0 / 64) * (BM * 128u) + row * 128u;
  const uint32_t chunk0 = static_cast<uint32_t>((c0 % 64) / 8);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t phys = (chunk0 + j) ^ (row & 7u);
    *reinterpret_cast<uint4*>(rowp + phys * 16u) = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  }
}

__global__ void __launch_bounds__(32 + 128 * kMaxWorkers, 1) mlp_fused_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const int E = p.workers;
  const Layout lo = make_layout(p.D, p.H, p.L, E);
  const uint32_t sbase = smem_u32(smem_raw);                     // small items
  const uint32_t base = (sbase + lo.small_bytes + 1023u) & ~1023u;  // swizzled buffers
  uint8_t* gbase = smem_raw + (base - sbase);
  const uint32_t warp = threadIdx.x / 32;
  const uint32_t lane = threadIdx.x % 32;
  const int num_tiles = (p.rows + BM - 1) / BM;

  const uint32_t w_full = sbase + lo.bar_off;
  auto x_full = [&](int g, int s) { return sbase + lo.bar_off + 8u * (1 + 2 * g + s); };
  auto slot_free = [&](int g, int s) { return sbase + lo.bar_off + 8u * (1 + 2 * E + 2 * g + s); };
  auto mma_done = [&](int g) { return sbase + lo.bar_off + 8u * (1 + 4 * E + g); };
  auto slot_addr = [&](int g, int s) { return lo.slot_off + static_cast<uint32_t>(2 * g + s) * lo.slot_bytes; };

  // ---- set-up: barriers, TMEM, biases (fp32), weights (TMA, once)
  if (threadIdx.x == 0) {
    mbar_init(w_full, 1);
    for (int g = 0; g < E; ++g) {
      for (int s = 0; s < 2; ++s) {
        mbar_init(x_full(g, s), 1);
        mbar_init(slot_free(g, s), 4);  // one arrival per warp of the worker
      }
      mbar_init(mma_done(g), 1);
    }
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(sbase + lo.tmem_slot_off, lo.tmem_cols);
    tmem_relinquish_alloc_permit();
  }
  float* bias_s = reinterpret_cast<float*>(smem_raw + lo.bias_off);
  for (int i = threadIdx.x; i < p.L * p.H; i += blockDim.x) {
    const int l = i / p.H, n = i % p.H;
    bias_s[i] = p.bias[l] != nullptr ? __half2float(__ushort_as_half(p.bias[l][n])) : 0.0f;
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem_raw + lo.tmem_slot_off);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&p.x_map);
      tma_prefetch_desc(&p.out_map);
      uint32_t wbytes = 0;
      for (int l = 0; l < p.L; ++l) wbytes += static_cast<uint32_t>(p.H / 64) * (l == 0 ? p.D : p.H) * 128u;
      mbar_arrive_expect_tx(w_full, wbytes);
      for (int l = 0; l < p.L; ++l) {
        const int K = l == 0 ? p.D : p.H;
        for (int j = 0; j < p.H / 64; ++j)
          tma_load_2d(base + lo.w_off[l] + static_cast<uint32_t>(j * K) * 128u, &p.w_map[l], w_full, j * 64, 0);
      }
      const uint32_t xbytes = static_cast<uint32_t>(p.D) * BM * 2u;
      int i = 0;
      for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++i) {
        const int g = i % E, n = i / E, s = n & 1, u = n >> 1;
        if (!mbar_wait(slot_free(g, s), (u & 1) ^ 1, p.err, kErrWaitMlp)) break;
        mbar_arrive_expect_tx(x_full(g, s), xbytes);
        for (int c = 0; c < p.D / 64; ++c)
          tma_load_2d(base + slot_addr(g, s) + static_cast<uint32_t>(c) * BM * 128u, &p.x_map, x_full(g, s), c * 64,
                      t * BM);
      }
      // Every issued load must land before the CTA may exit.
      mbar_wait(w_full, 0, p.err, kErrWaitMlp);
      const int issued = i;
      for (int k = issued - 1; k >= 0 && k >= issued - 2 * E; --k) {
        const int g = k % E, n = k / E;
        mbar_wait(x_full(g, n & 1), (n >> 1) & 1, p.err, kErrWaitMlp);
      }
    }
  } else {
    // ------------------------------------------------------------ row-tile workers
    const int g = static_cast<int>(warp - 1) / 4;
    if (g < E) {
      const uint32_t q = warp & 3u;               // TMEM lane quarter of this warp
      const uint32_t row = 32u * q + lane;        // row within the tile (= TMEM lane)
      const bool leader = (warp == static_cast<uint32_t>(1 + 4 * g)) && lane == 0;
      const uint32_t tmem_acc = tmem_base + static_cast<uint32_t>(g * p.H);
      const uint32_t tmem_row = tmem_acc + ((32u * q) << 16);
      const uint32_t bar_id = 1u + static_cast<uint32_t>(g);
      uint32_t mma_phase = 0;
      bool ok = mbar_wait(w_full, 0, p.err, kErrWaitMlp);
      int n = 0;
      int pending_free = -1;  // slot whose output store must finish before it is handed back
      for (int t = blockIdx.x + g * gridDim.x; ok && t < num_tiles; t += E * gridDim.x, ++n) {
        const int s = n & 1, u = n >> 1;
        if (!mbar_wait(x_full(g, s), u & 1, p.err, kErrWaitMlp)) {
          ok = false;
          break;
        }
        uint8_t* slot = gbase + slot_addr(g, s);
        const uint32_t slot_a = base + slot_addr(g, s);
        for (int l = 0; l < p.L; ++l) {
          const int K = l == 0 ? p.D : p.H;
          if (leader) {
            tc_fence_after_sync();
            const uint32_t idesc = idesc_f16_f32acc(false, false, true, BM, static_cast<uint32_t>(p.H));
            const uint32_t wa = base + lo.w_off[l];
            for (int ks = 0; ks < K / 16; ++ks) {
              const uint64_t ad =
                  smem_desc_sw128(slot_a + static_cast<uint32_t>(ks / 4) * BM * 128u + (ks % 4) * 32u, 16, 1024);
              const uint64_t bd = smem_desc_sw128(wa + static_cast<uint32_t>(ks) * 2048u,
                                                  static_cast<uint32_t>(K) * 128u, 1024);
              tc_mma_f16(tmem_acc, ad, bd, idesc, ks > 0 ? 1u : 0u);
            }
            tc_commit(mma_done(g));
          }
          if (l == 0 && pending_free >= 0) {
            // The previous tile's output store has had a whole MMA to read its slot.
            if (lane == 0) {
              bulk_wait_group_read<0>();
              mbar_arrive(slot_free(g, pending_free));
            }
            pending_free = -1;
          }
          if (!mbar_wait(mma_done(g), mma_phase, p.err, kErrWaitMlp)) {
            ok = false;
            break;
          }
          mma_phase ^= 1u;
          tc_fence_after_sync();
          const float* bl = bias_s + l * p.H;
          const bool last = (l == p.L - 1);
          const int act = last ? kActNone : p.act;
          for (int c0 = 0; c0 < p.H; c0 += 32) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(tmem_row + static_cast<uint32_t>(c0), r);
            tmem_ld_wait();
            switch (act) {
              case kActSoftplus:
                epilogue_cols32<kActSoftplus>(r, bl, c0, slot, row);
                break;
              case kActRelu:
                epilogue_cols32<kActRelu>(r, bl, c0, slot, row);
                break;
              case kActGeluErf:
                epilogue_cols32<kActGeluErf>(r, bl, c0, slot, row);
                break;
              default:
                epilogue_cols32<kActNone>(r, bl, c0, slot, row);
                break;
            }
          }
          // TMEM reads done and the slot rewritten: publish to the tensor core / TMA.
          tc_fence_before_sync();
          fence_proxy_async_smem();
          named_bar_sync(bar_id, 128);
        }
        if (!ok) break;
        // This warp's 32 rows of the finished tile go out by TMA.
        if (lane == 0) {
          for (int c = 0; c < p.H / 64; ++c)
            tma_store_2d(&p.out_map, slot_a + static_cast<uint32_t>(c) * BM * 128u + 32u * q * 128u, c * 64,
                         t * BM + static_cast<int>(32u * q));
          bulk_commit_group();
        }
        pending_free = s;
      }
      if (lane == 0) bulk_wait_group<0>();
      __syncwarp();
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, lo.tmem_cols);
  }
}

}  // namespace mlp

uint32_t mlp_max_weight_bytes() { return mlp::kWeightBudget; }

cudaError_t launch_mlp_fused(const DeviceCtx& dev, int64_t rows, int D, int H, int L, const void* x,
                             const void* const* W, const void* const* b, void* out, int act, cudaStream_t stream) {
  using namespace mlp;
  if (L > kMaxLayers || D % 64 != 0 || H % 64 != 0) return cudaErrorNotSupported;
  // Largest number of row-tile workers that fits shared memory and TMEM.
  int E = 0;
  for (int e = kMaxWorkers; e >= 1; --e) {
    const Layout lo = make_layout(D, H, L, e);
    if (lo.alloc_bytes <= kSmemLimit && e * H <= 512) {
      E = e;
      break;
    }
  }
  if (E == 0) return cudaErrorNotSupported;
  const Layout lo = make_layout(D, H, L, E);
  const uint32_t smem = lo.alloc_bytes;

  Params p;
  memset(&p, 0, sizeof(p));
  cudaError_t e;
  if ((e = encode_tmap_2d(&p.x_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, x, rows, D, BM, 64,
                          CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return e;
  if ((e = encode_tmap_2d(&p.out_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, out, rows, H, 32, 64,
                          CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return e;
  for (int l = 0; l < L; ++l) {
    const int K = l == 0 ? D : H;
    if ((e = encode_tmap_2d(&p.w_map[l], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, W[l], K, H, K, 64,
                            CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
      return e;
    p.bias[l] = b != nullptr ? static_cast<const uint16_t*>(b[l]) : nullptr;
  }
  p.rows = static_cast<int>(rows);
  p.D = D;
  p.H = H;
  p.L = L;
  p.act = act;
  p.workers = E;
  p.err = dev.err_word;

  if ((e = cudaFuncSetAttribute(mlp_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
    return e;
  const int64_t tiles = (rows + BM - 1) / BM;
  const int grid = static_cast<int>(tiles < dev.sm_count ? tiles : dev.sm_count);
  const int threads = 32 + 128 * E;
  mlp_fused_kernel<<<grid, threads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace coalesce
