// The general form of the tcgen05 GEMM (gemm_tc.cu) for the backward pass of
// the chained MLP (the "MLP Megakernel" README, "Key ideas": above 32K rows
// the weight gradients come from GEMMs interleaved with the data-gradient
// computation).  Same tile shape, warp roles, stage ring and double-buffered
// TMEM accumulators as the forward kernel, plus:
//   * kTransA: A is given as At [K, M] row-major and read as an MN-major
//     operand (two [64 k x 64 m] boxes per stage), so dW = h^T g needs no
//     transposed copy of h;
//   * kTransB: B is given as Bt [N, K] row-major and read K-major (one
//     [256 n x 64 k] box per stage), so g W^T reads W as stored;
//   * kMode 1: Y is fp32 and the tile is added into it (TMA reduce-add), and
//     the K range is split over several CTAs: the weight gradients have
//     K = rows (up to millions) but only one or two output tiles;
//   * kMode 2: Y = (A B) * act'(aux), aux being the activation's output h:
//     the data gradient through softplus (act' = 1 - e^-h) or ReLU.
#include "gemm_tc.cuh"

namespace coalesce {
namespace tcgemm {

constexpr int kModeStore = 0;   // Y (16-bit) = act(A B + bias)
constexpr int kModeAccF32 = 1;  // Y (fp32) += A B, K split over CTAs
constexpr int kModeDAct = 2;    // Y (16-bit) = (A B) * act'(aux)

// This lane's aux values for a 64-column slice: row `row`, columns n0 .. n0+63
// of the 16-bit [M, N] matrix, as eight 16-byte loads (zero outside it).
__device__ __forceinline__ void load_aux8(const uint16_t* __restrict__ aux, int row, int M, int n0, int N,
                                          uint4* dst) {
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const int nc = n0 + 8 * g;
    dst[g] = (row < M && nc < N) ? __ldg(reinterpret_cast<const uint4*>(aux + static_cast<size_t>(row) * N + nc))
                                 : make_uint4(0u, 0u, 0u, 0u);
  }
}

// One 32-row x 64-column slice of (A B) * act'(aux) into the swizzled staging
// buffer; `av` holds this lane's aux values for the slice (load_aux8).
template <bool kBF16, int kAct>
__device__ __forceinline__ void dact_slice(const uint32_t* r, const uint4* av, uint8_t* buf, uint32_t lane) {
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    float hv[8];
    unpack8(av[g], kBF16, hv);
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float y0 = __uint_as_float(r[8 * g + 2 * i]) * dact_from_output<kAct>(hv[2 * i]);
      const float y1 = __uint_as_float(r[8 * g + 2 * i + 1]) * dact_from_output<kAct>(hv[2 * i + 1]);
      w[i] = pack2(y0, y1, kBF16);
    }
    const uint32_t chunk = static_cast<uint32_t>(g) ^ (lane & 7u);
    *reinterpret_cast<uint4*>(buf + lane * 128u + chunk * 16u) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// 32 fp32 accumulator columns of row `lane` into a 32 x 32 fp32 staging box
// (128-B rows, 16-B chunk j at j ^ (lane & 7)).
__device__ __forceinline__ void f32_slice(const uint32_t* r, uint8_t* buf, uint32_t lane) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t chunk = static_cast<uint32_t>(j) ^ (lane & 7u);
    *reinterpret_cast<uint4*>(buf + lane * 128u + chunk * 16u) =
        make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
  }
}

// The general form (transposed operands, fp32 accumulation, derivative
// epilogue) for the MLP's backward; the plain store path is kept as its own
// kernel (gemm_tc.cu) so that these options do not touch the forward GEMM.
template <bool kBF16, bool kTransA, bool kTransB, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_ex_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                            const __grid_constant__ CUtensorMap tmap_y, const uint16_t* __restrict__ bias,
                            const uint16_t* __restrict__ aux, int M, int N, int K, int act, int splits,
                            uint32_t* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_addr);

  const uint32_t warp = warp_index_uniform();
  const uint32_t lane = threadIdx.x % 32;
  const int num_m = (M + BM - 1) / BM;
  const int num_n = (N + BN - 1) / BN;
  const int num_kb = (K + BK - 1) / BK;
  const int num_tiles = num_m * num_n;
  // Work unit u: output tile u / splits, k blocks [kb_lo(u), kb_hi(u)).
  const int num_units = num_tiles * splits;
  auto kb_lo = [&](int u) {
    return splits == 1 ? 0 : static_cast<int>(static_cast<int64_t>(u % splits) * num_kb / splits);
  };
  auto kb_hi = [&](int u) {
    return splits == 1 ? num_kb : static_cast<int>(static_cast<int64_t>(u % splits + 1) * num_kb / splits);
  };

  const uint32_t bar0 = base + kOffBars;
  auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
  auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (STAGES + s); };
  auto accf_bar = [&](uint32_t a) { return bar0 + 8u * (2 * STAGES + a); };
  auto acce_bar = [&](uint32_t a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
  const uint32_t mma_done_bar = bar0 + 8u * (2 * STAGES + 4);

  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (uint32_t a = 0; a < 2; ++a) {
      mbar_init(accf_bar(a), 1);
      mbar_init(acce_bar(a), kEpiWarps);
    }
    mbar_init(mma_done_bar, 1);
    fence_mbarrier_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
    tma_prefetch_desc(&tmap_y);
  }
  if (warp == 1) {
    tmem_alloc(base + kOffTmemSlot, kTmemCols);
    tmem_relinquish_alloc_permit();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(gbase + kOffTmemSlot);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int issued = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
        int mb, nb;
        tile_coords(splits == 1 ? u : u / splits, num_m, num_n, mb, nb);
        const int kb_end = kb_hi(u);
        for (int kb = kb_lo(u); kb < kb_end; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, err, kErrWaitProducer)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, kABytes + kBBytes);
          if constexpr (kTransA) {
            // At [K, M]: two [64 k x 64 m] MN-major boxes
#pragma unroll
            for (int j = 0; j < BM / 64; ++j)
              tma_load_2d(base + kOffA + stage * kABytes + j * kBChunkBytes, &tmap_a, fb, mb * BM + j * 64, kb * BK);
          } else {
            tma_load_2d(base + kOffA + stage * kABytes, &tmap_a, fb, kb * BK, mb * BM);
          }
          if constexpr (kTransB) {
            // Bt [N, K]: one [256 n x 64 k] K-major box
            tma_load_2d(base + kOffB + stage * kBBytes, &tmap_b, fb, kb * BK, nb * BN);
          } else {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j) {
              tma_load_2d(base + kOffB + stage * kBBytes + j * kBChunkBytes, &tmap_b, fb, nb * BN + j * 64, kb * BK);
            }
          }
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Before the CTA can exit, every TMA load it issued must have landed.
      // (Already true on the normal path; matters only after a timeout.)
      for (int i = 0; i < STAGES && i < issued; ++i) {
        if (stage == 0) {
          stage = STAGES - 1;
          phase ^= 1u;
        } else {
          --stage;
        }
        mbar_wait(full_bar(stage), phase, err, kErrWaitProducer);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32acc(kBF16, kTransA, !kTransB, BM, BN);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
        if (!mbar_wait(acce_bar(acc), acc_phase ^ 1u, err, kErrWaitMma)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * BN;
        const int kb0 = kb_lo(u);
        const int kb_end = kb_hi(u);
        for (int kb = kb0; kb < kb_end; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, err, kErrWaitMma)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a_addr = base + kOffA + stage * kABytes;
          const uint32_t b_addr = base + kOffB + stage * kBBytes;
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks) {
            const uint64_t ad = kTransA ? smem_desc_sw128(a_addr + ks * 2048, kBChunkBytes, 1024)
                                        : smem_desc_sw128(a_addr + ks * 32, 16, 1024);
            const uint64_t bd = kTransB ? smem_desc_sw128(b_addr + ks * 32, 16, 1024)
                                        : smem_desc_sw128(b_addr + ks * 2048, kBChunkBytes, 1024);
            tc_mma_f16(d_tmem, ad, bd, idesc, (kb != kb0 || ks != 0) ? 1u : 0u);
          }
          tc_commit(empty_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(accf_bar(acc));
        acc ^= 1u;
        if (acc == 0) acc_phase ^= 1u;
      }
      // All MMAs issued by this thread are complete once this commit arrives.
      tc_commit(mma_done_bar);
      mbar_wait(mma_done_bar, 0, err, kErrWaitMma);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const uint32_t q = warp & 3u;          // TMEM lane quarter this warp may access
    const uint32_t ew = warp - 2u;         // staging-buffer owner index
    uint8_t* out_buf0 = gbase + kOffOut + ew * 2u * kOutBufBytes;
    const uint32_t out_addr0 = base + kOffOut + ew * 2u * kOutBufBytes;
    uint32_t acc = 0, acc_phase = 0, ob = 0;
    // kModeDAct: the aux values of the next slice are loaded one slice ahead
    // (across tiles too), so their memory latency overlaps this slice's work.
    uint4 aux_next[8];
    if constexpr (kMode == kModeDAct) {
      if (static_cast<int>(blockIdx.x) < num_units) {
        int mb, nb;
        tile_coords(static_cast<int>(blockIdx.x), num_m, num_n, mb, nb);
        load_aux8(aux, mb * BM + 32 * static_cast<int>(q) + static_cast<int>(lane), M, nb * BN, N, aux_next);
      }
    }
    for (int u = blockIdx.x; u < num_units; u += gridDim.x) {
      int mb, nb;
      tile_coords(splits == 1 ? u : u / splits, num_m, num_n, mb, nb);
      if (!mbar_wait(accf_bar(acc), acc_phase, err, kErrWaitEpilogue)) break;
      tc_fence_after_sync();
      const int row0 = mb * BM + 32 * static_cast<int>(q);
      const int n_left = N - nb * BN;
      const int nslices = min(BN / 64, (n_left + 63) / 64);
#pragma unroll 1
      for (int c = 0; c < nslices; ++c) {
        uint4 aux_cur[8];
        if constexpr (kMode == kModeDAct) {
#pragma unroll
          for (int g = 0; g < 8; ++g) aux_cur[g] = aux_next[g];
          if (c + 1 < nslices) {
            load_aux8(aux, row0 + static_cast<int>(lane), M, nb * BN + (c + 1) * 64, N, aux_next);
          } else if (u + static_cast<int>(gridDim.x) < num_units) {
            int mb2, nb2;
            tile_coords(u + static_cast<int>(gridDim.x), num_m, num_n, mb2, nb2);
            load_aux8(aux, mb2 * BM + 32 * static_cast<int>(q) + static_cast<int>(lane), M, nb2 * BN, N, aux_next);
          }
        }
        uint32_t r[64];
        const uint32_t taddr = tmem_base + ((32u * q) << 16) + acc * BN + c * 64;
        tmem_ld_32x32b_x32(taddr, r);
        tmem_ld_32x32b_x32(taddr + 32, r + 32);
        tmem_ld_wait();
        if (c == nslices - 1) {
          // This warp has read its whole share of the accumulator: hand it back.
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(acce_bar(acc));
        }
        const int n0 = nb * BN + c * 64;
        if constexpr (kMode == kModeAccF32) {
          // fp32 tile added into Y: two 32-column boxes per slice
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            if (lane == 0) bulk_wait_group_read<1>();
            __syncwarp();
            f32_slice(r + 32 * h, out_buf0 + ob * kOutBufBytes, lane);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_reduce_add_2d(&tmap_y, out_addr0 + ob * kOutBufBytes, n0 + 32 * h, row0);
              bulk_commit_group();
            }
            ob ^= 1u;
          }
          continue;
        }
        // The TMA store issued from this buffer two slices ago must have read it.
        if (lane == 0) bulk_wait_group_read<1>();
        __syncwarp();
        uint8_t* buf = out_buf0 + ob * kOutBufBytes;
        if constexpr (kMode == kModeDAct) {
          switch (act) {
            case kActSoftplus:
              dact_slice<kBF16, kActSoftplus>(r, aux_cur, buf, lane);
              break;
            case kActRelu:
              dact_slice<kBF16, kActRelu>(r, aux_cur, buf, lane);
              break;
            default:
              dact_slice<kBF16, kActNone>(r, aux_cur, buf, lane);
              break;
          }
        } else {
          switch (act) {
            case kActRelu:
              epilogue_slice<kBF16, kActRelu>(r, bias, n0, N, buf, lane);
              break;
            case kActGeluErf:
              epilogue_slice<kBF16, kActGeluErf>(r, bias, n0, N, buf, lane);
              break;
            case kActSoftplus:
              epilogue_slice<kBF16, kActSoftplus>(r, bias, n0, N, buf, lane);
              break;
            default:
              epilogue_slice<kBF16, kActNone>(r, bias, n0, N, buf, lane);
              break;
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(&tmap_y, out_addr0 + ob * kOutBufBytes, n0, row0);
          bulk_commit_group();
        }
        ob ^= 1u;
      }
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace tcgemm

namespace {

template <bool kBF16, bool kTA, bool kTB>
void (*pick_kernel(int mode))(CUtensorMap, CUtensorMap, CUtensorMap, const uint16_t*, const uint16_t*, int, int, int,
                              int, int, uint32_t*) {
  using namespace tcgemm;
  switch (mode) {
    case kModeAccF32:
      return gemm_tc_ex_kernel<kBF16, kTA, kTB, kModeAccF32>;
    case kModeDAct:
      return gemm_tc_ex_kernel<kBF16, kTA, kTB, kModeDAct>;
    default:
      return gemm_tc_ex_kernel<kBF16, kTA, kTB, kModeStore>;
  }
}

}  // namespace

cudaError_t launch_gemm_tc_ex(const DeviceCtx& dev, bool bf16, bool trans_a, bool trans_b, int mode, int64_t M,
                              int64_t N, int64_t K, const void* A, const void* B, const void* bias, const void* aux,
                              void* Y, int act, cudaStream_t stream) {
  using namespace tcgemm;
  if (!trans_a && !trans_b && mode == kModeStore) return launch_gemm_tc(dev, bf16, M, N, K, A, B, bias, Y, act, stream);
  const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap ta, tb, ty;
  cudaError_t e;
  if (trans_a) {
    e = encode_tmap_2d(&ta, dt, 2, A, K, M, BK, 64, CU_TENSOR_MAP_SWIZZLE_128B);  // At [K, M]
  } else {
    e = encode_tmap_2d(&ta, dt, 2, A, M, K, BM, BK, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (e != cudaSuccess) return e;
  if (trans_b) {
    e = encode_tmap_2d(&tb, dt, 2, B, N, K, BN, BK, CU_TENSOR_MAP_SWIZZLE_128B);  // Bt [N, K]
  } else {
    e = encode_tmap_2d(&tb, dt, 2, B, K, N, BK, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (e != cudaSuccess) return e;
  if (mode == kModeAccF32) {
    e = encode_tmap_2d(&ty, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, Y, M, N, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    e = encode_tmap_2d(&ty, dt, 2, Y, M, N, 32, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (e != cudaSuccess) return e;

  using Kernel = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, const uint16_t*, const uint16_t*, int, int, int, int,
                          int, uint32_t*);
  Kernel kernel;
  if (bf16) {
    kernel = trans_a ? (trans_b ? pick_kernel<true, true, true>(mode) : pick_kernel<true, true, false>(mode))
                     : (trans_b ? pick_kernel<true, false, true>(mode) : pick_kernel<true, false, false>(mode));
  } else {
    kernel = trans_a ? (trans_b ? pick_kernel<false, true, true>(mode) : pick_kernel<false, true, false>(mode))
                     : (trans_b ? pick_kernel<false, false, true>(mode) : pick_kernel<false, false, false>(mode));
  }
  if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes)) != cudaSuccess)
    return e;
  const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  const int64_t num_kb = (K + BK - 1) / BK;
  // The fp32-accumulate mode splits K until every SM has a work unit (each
  // unit keeps at least 4 k blocks); the other modes own whole tiles.
  int64_t splits = 1;
  if (mode == kModeAccF32) {
    while (tiles * splits * 2 <= dev.sm_count && splits * 2 * 4 <= num_kb) splits *= 2;
    if (tiles * splits < dev.sm_count) {
      const int64_t want = (dev.sm_count + tiles - 1) / tiles;
      splits = want * 4 <= num_kb ? want : (num_kb / 4 > splits ? num_kb / 4 : splits);
    }
  }
  const int64_t units = tiles * splits;
  const int grid = static_cast<int>(units < dev.sm_count ? units : dev.sm_count);
  kernel<<<grid, kThreads, kSmemBytes, stream>>>(ta, tb, ty, static_cast<const uint16_t*>(bias),
                                                 static_cast<const uint16_t*>(aux), static_cast<int>(M),
                                                 static_cast<int>(N), static_cast<int>(K), act,
                                                 static_cast<int>(splits), dev.err_word);
  return cudaGetLastError();
}

}  // namespace coalesce
