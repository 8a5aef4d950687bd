// fp16 / bf16 GEMM with a fused bias + activation epilogue on the tcgen05
// tensor cores (sm_103a).
//
//   Y[M, N] = act(A[M, K] . B[K, N] + bias[N]),   fp32 accumulation in TMEM.
//
// The operation is the fused GEMM + bias + GELU of the "Coalesce" README
// ("Fusion study (03_matmul_fused)"): the bias-add and activation run on the
// accumulator before the one and only store of Y, so no unfused intermediate
// ever reaches memory (the "Fuse Elementwise Ops" page, "Handle epilogue
// fusion into GEMM/conv separately" and the traffic count in step 2).
//
// Design (one CTA per SM, persistent over output tiles):
//   warp 0      TMA producer: A tile [128 x 64] (K-major, 128-B swizzle) and
//               B tile [64 x 256] as four [64 k x 64 n] MN-major chunks into a
//               4-stage shared-memory ring, completion on mbarriers.
//   warp 1      allocates 512 TMEM columns (two 128 x 256 fp32 accumulators)
//               and, from one lane, issues tcgen05.mma (M=128, N=256, K=16)
//               and tcgen05.commit to release stages / publish accumulators.
//   warps 2..5  epilogue: tcgen05.ld a 32-row x 64-column slice, add the bias,
//               apply the activation in fp32, round to fp16/bf16 (RNE), stage
//               through a 128-B-swizzled shared buffer and TMA-store it.  The
//               double-buffered accumulators let the epilogue of tile i run
//               while the tensor cores compute tile i+1.
// Tiles are visited in groups of 32 row-blocks so that concurrently running
// CTAs share A and B panels in L2 (the "MLP Megakernel" README, GROUP_M):
// for the 16384 x 16384 x 4096 GEMM a group's A panel (32 MiB) stays in L2
// while B streams once per group; 16 and 64 were slower (measured).
// Ragged M, N and K tails are handled by TMA: loads zero-fill outside the
// matrix and stores clip to it.  Problems that give every SM pair a 256 x 256
// tile run on CTA pairs instead (gemm_tc_pair.cu).
#include "gemm_tc.cuh"

namespace coalesce {
namespace tcgemm {

template <bool kBF16>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_bias_act_tc_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                            const __grid_constant__ CUtensorMap tmap_y, const uint16_t* __restrict__ bias, int M,
                            int N, int K, int act, uint32_t* err) {
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
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        int mb, nb;
        tile_coords(t, num_m, num_n, mb, nb);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, err, kErrWaitProducer)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, kABytes + kBBytes);
          tma_load_2d(base + kOffA + stage * kABytes, &tmap_a, fb, kb * BK, mb * BM);
#pragma unroll
          for (int j = 0; j < BN / 64; ++j) {
            tma_load_2d(base + kOffB + stage * kBBytes + j * kBChunkBytes, &tmap_b, fb, nb * BN + j * 64, kb * BK);
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
      constexpr uint32_t idesc = idesc_f16_f32acc(kBF16, false, true, BM, BN);
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
        if (!mbar_wait(acce_bar(acc), acc_phase ^ 1u, err, kErrWaitMma)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, err, kErrWaitMma)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t a_addr = base + kOffA + stage * kABytes;
          const uint32_t b_addr = base + kOffB + stage * kBBytes;
#pragma unroll
          for (int ks = 0; ks < BK / 16; ++ks) {
            const uint64_t ad = smem_desc_sw128(a_addr + ks * 32, 16, 1024);
            const uint64_t bd = smem_desc_sw128(b_addr + ks * 2048, kBChunkBytes, 1024);
            tc_mma_f16(d_tmem, ad, bd, idesc, (kb | ks) != 0 ? 1u : 0u);
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
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      int mb, nb;
      tile_coords(t, num_m, num_n, mb, nb);
      if (!mbar_wait(accf_bar(acc), acc_phase, err, kErrWaitEpilogue)) break;
      tc_fence_after_sync();
      const int row0 = mb * BM + 32 * static_cast<int>(q);
      const int n_left = N - nb * BN;
      const int nslices = min(BN / 64, (n_left + 63) / 64);
#pragma unroll 1
      for (int c = 0; c < nslices; ++c) {
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
        // The TMA store issued from this buffer two slices ago must have read it.
        if (lane == 0) bulk_wait_group_read<1>();
        __syncwarp();
        uint8_t* buf = out_buf0 + ob * kOutBufBytes;
        const int n0 = nb * BN + c * 64;
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

cudaError_t launch_gemm_tc(const DeviceCtx& dev, bool bf16, int64_t M, int64_t N, int64_t K, const void* A,
                           const void* B, const void* bias, void* Y, int act, cudaStream_t stream) {
  using namespace tcgemm;
  // Problems that give every SM pair a 256 x 256 tile go to the CTA-pair
  // kernel (gemm_tc_pair.cu).
  if (gemm_tc_pair_supported(M, N, K) && ((M + 255) / 256) * ((N + 255) / 256) >= dev.sm_count / 2) {
    const cudaError_t e = launch_gemm_tc_pair(dev, bf16, M, N, K, A, B, bias, Y, act, stream);
    if (e != cudaErrorNotSupported) return e;
  }
  const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap ta, tb, ty;
  cudaError_t e;
  if ((e = encode_tmap_2d(&ta, dt, 2, A, M, K, BM, BK, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess) return e;
  if ((e = encode_tmap_2d(&tb, dt, 2, B, K, N, BK, 64, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess) return e;
  if ((e = encode_tmap_2d(&ty, dt, 2, Y, M, N, 32, 64, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess) return e;

  auto kernel = bf16 ? gemm_bias_act_tc_kernel<true> : gemm_bias_act_tc_kernel<false>;
  if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes)) != cudaSuccess)
    return e;
  const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  const int grid = static_cast<int>(tiles < dev.sm_count ? tiles : dev.sm_count);
  kernel<<<grid, kThreads, kSmemBytes, stream>>>(ta, tb, ty, static_cast<const uint16_t*>(bias), static_cast<int>(M),
                                                 static_cast<int>(N), static_cast<int>(K), act, dev.err_word);
  return cudaGetLastError();
}

}  // namespace coalesce
