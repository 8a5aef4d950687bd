// fp16 / bf16 GEMM + bias + activation on CTA pairs: the same operation as
// gemm_tc.cu,
//
//   Y[M, N] = act(A[M, K] . B[K, N] + bias[N]),   fp32 accumulation in TMEM,
//
// with each 256 x 256 output tile computed by two CTAs on two SMs through the
// tensor cores' pair form (tcgen05.mma.cta_group::2).  Each CTA holds 128 rows
// of A and 128 of the tile's 256 columns of B per k step; one MMA instruction
// of the even CTA covers the pair, and each CTA's TMEM receives its own 128
// rows x 256 columns.  Compared with one CTA per 128 x 256 tile, a pipeline
// stage needs 32 KiB of shared memory instead of 48 KiB, so the ring holds six
// stages instead of four, the MMAs read a third less shared memory per
// k step, and one issuing thread serves two SMs.
//
// Per CTA (one per SM, persistent over pair tiles):
//   warp 0      TMA producer: this CTA's A rows [128 x 64] and B columns
//               [64 x 128] (two MN-major 64-column chunks) of each k step into
//               its own ring.  Both CTAs' loads complete on the even CTA's
//               full barrier (the TMA's pair form), which expects both CTAs'
//               bytes.
//   warp 1      even CTA: issues the pair MMAs (M = 256, N = 256, K = 16)
//               once a stage is full and commits them to both CTAs' empty and
//               accumulator barriers.  Both CTAs' warp 1 allocate the pair's
//               512 TMEM columns.
//   warps 2..5  epilogue, as in gemm_tc.cu, on this CTA's 128 rows; the
//               release of an accumulator is an arrive on the even CTA's
//               barrier (local or remote).
// Tiles are visited in groups of 16 pair rows (4096 rows of A in L2, as with
// 32 row blocks of 128 in gemm_tc.cu).  Ragged edges: TMA zero-fills boxes
// that straddle the matrix and clips stores; a box that would start beyond
// it (the odd CTA's rows of a last pair row, a last B chunk) is not loaded at
// all, and stores of rows beyond M are skipped.
#include "gemm_tc.cuh"
#include "sm100_pair.cuh"

#include <atomic>

namespace coalesce {
namespace tcpair {

constexpr int PM = 256;  // rows per pair tile (128 per CTA)
constexpr int HM = 128;  // rows per CTA
constexpr int PN = 256;  // columns per pair tile
constexpr int BK = 64;
constexpr int STAGES = 6;
constexpr int kEpiWarps = 4;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kGroupPairs = 16;

constexpr uint32_t kABytes = HM * BK * 2;         // 16 KiB
constexpr uint32_t kBChunkBytes = BK * 64 * 2;    // 8 KiB: 64 k-rows x 64 n (128 B)
constexpr uint32_t kBBytes = BK * (PN / 2) * 2;   // 16 KiB: this CTA's 128 columns
constexpr uint32_t kOutBufBytes = 32 * 64 * 2;    // 32 rows x 64 cols
constexpr uint32_t kTmemCols = 2 * PN;

constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffB = kOffA + STAGES * kABytes;
constexpr uint32_t kOffOut = kOffB + STAGES * kBBytes;
constexpr uint32_t kOffBars = kOffOut + kEpiWarps * 2 * kOutBufBytes;
constexpr uint32_t kNumBars = 2 * STAGES + 4 + 1;  // full, empty, acc_full x2, acc_empty x2, mma_done
constexpr uint32_t kOffTmemSlot = kOffBars + kNumBars * 8;
constexpr uint32_t kSmemBytes = kOffTmemSlot + 16 + 1024;  // + slack to align the base to 1 KiB

static_assert(kSmemBytes <= 232448, "shared memory budget exceeded");

// 64-column chunks of B that start inside N, of the two a CTA loads from column `col`.
__device__ __forceinline__ int b_chunks_in(int col, int N) { return col >= N ? 0 : min(2, (N - col + 63) / 64); }

__device__ __forceinline__ void pair_tile_coords(int t, int num_m, int num_n, int& mb, int& nb) {
  const int per_group = kGroupPairs * num_n;
  const int group = t / per_group;
  const int first_m = group * kGroupPairs;
  const int gm = min(num_m - first_m, kGroupPairs);
  const int r = t - group * per_group;
  mb = first_m + r % gm;
  nb = r / gm;
}

template <bool kBF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_bias_act_tc_pair_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                                 const __grid_constant__ CUtensorMap tmap_y, const uint16_t* __restrict__ bias, int M,
                                 int N, int K, int act, uint32_t* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw_addr);

  const uint32_t warp = warp_index_uniform();
  const uint32_t lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();  // 0: issues the pair's MMAs
  const int num_m = (M + PM - 1) / PM;
  const int num_n = (N + PN - 1) / PN;
  const int num_kb = (K + BK - 1) / BK;
  const int num_tiles = num_m * num_n;
  const int pair = static_cast<int>(blockIdx.x) >> 1;
  const int num_pairs = static_cast<int>(gridDim.x) >> 1;

  const uint32_t bar0 = base + kOffBars;
  auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
  auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (STAGES + s); };
  auto accf_bar = [&](uint32_t a) { return bar0 + 8u * (2 * STAGES + a); };
  auto acce_bar = [&](uint32_t a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
  const uint32_t mma_done_bar = bar0 + 8u * (2 * STAGES + 4);

  if (threadIdx.x == 0) {
    for (uint32_t s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);  // used on the even CTA only
      mbar_init(empty_bar(s), 1);
    }
    for (uint32_t a = 0; a < 2; ++a) {
      mbar_init(accf_bar(a), 1);
      mbar_init(acce_bar(a), 2 * kEpiWarps);  // both CTAs' epilogue warps (used on the even CTA)
    }
    mbar_init(mma_done_bar, 1);
    fence_mbarrier_init();
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
    tma_prefetch_desc(&tmap_y);
  }
  if (warp == 1) {
    tmem_alloc_pair(base + kOffTmemSlot, kTmemCols);
    tmem_relinquish_alloc_permit_pair();
  }
  tc_fence_before_sync();
  __syncthreads();
  // Both CTAs' barriers are initialised before either CTA signals the other's.
  cluster_sync_all();
  tc_fence_after_sync();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(gbase + kOffTmemSlot);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int issued = 0;
      bool ok = true;
      for (int t = pair; t < num_tiles && ok; t += num_pairs) {
        int mb, nb;
        pair_tile_coords(t, num_m, num_n, mb, nb);
        const int row = mb * PM + static_cast<int>(rank) * HM;       // this CTA's rows of A
        const int col = nb * PN + static_cast<int>(rank) * (PN / 2);  // this CTA's columns of B
        // Boxes that would start beyond the matrix are not loaded: their rows
        // or columns of the tile are never stored, so whatever the stage
        // holds there only reaches discarded accumulator entries.  The even
        // CTA's barrier expects the bytes of the boxes both CTAs do load.
        const bool a_in = row < M;
        const int b_in = b_chunks_in(col, N);
        uint32_t pair_bytes = 0;
        for (int r = 0; r < 2; ++r)
          pair_bytes += (mb * PM + r * HM < M ? kABytes : 0u) +
                        static_cast<uint32_t>(b_chunks_in(nb * PN + r * (PN / 2), N)) * kBChunkBytes;
        for (int kb = 0; kb < num_kb; ++kb) {
          // freed by the even CTA's MMA commit
          if (!mbar_wait_cluster(empty_bar(stage), phase ^ 1u, err, kErrWaitProducer)) {
            ok = false;
            break;
          }
          // the even CTA's full barrier, which counts both CTAs' bytes
          const uint32_t fb = mapa_shared(full_bar(stage), 0);
          if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), pair_bytes);
          if (a_in) tma_load_2d_pair(base + kOffA + stage * kABytes, &tmap_a, fb, kb * BK, row);
          for (int j = 0; j < b_in; ++j)
            tma_load_2d_pair(base + kOffB + stage * kBBytes + j * kBChunkBytes, &tmap_b, fb, col + j * 64, kb * BK);
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Before the pair can exit, every TMA load it issued must have landed
      // (already true on the normal path; matters only after a timeout).  The
      // even CTA's full barriers count both CTAs' loads; the odd CTA leaves
      // only after the even one (final cluster barrier).
      for (int i = 0; rank == 0 && i < STAGES && i < issued; ++i) {
        if (stage == 0) {
          stage = STAGES - 1;
          phase ^= 1u;
        } else {
          --stage;
        }
        mbar_wait_cluster(full_bar(stage), phase, err, kErrWaitProducer);
      }
      // After a timeout the odd CTA may have issued a stage the even CTA never
      // armed, so no barrier it can wait on tracks that load (a CTA can only
      // wait on its own barriers).  It waits out a fixed 200 us instead, far
      // longer than a 32 KiB tile load takes, before the pair may exit.
      if (rank == 1 && !ok) {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
      }
    }
  } else if (warp == 1) {
    if (rank == 0) {
      // ---------------------------------------------------------- MMA issuer (even CTA)
      if (lane == 0) {
        constexpr uint32_t idesc = idesc_f16_f32acc(kBF16, false, true, PM, PN);
        uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
        bool ok = true;
        for (int t = pair; t < num_tiles && ok; t += num_pairs) {
          // both CTAs' epilogues have read this accumulator
          if (!mbar_wait_cluster(acce_bar(acc), acc_phase ^ 1u, err, kErrWaitMma)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t d_tmem = tmem_base + acc * PN;
          for (int kb = 0; kb < num_kb; ++kb) {
            // both CTAs' halves of the stage have landed
            if (!mbar_wait_cluster(full_bar(stage), phase, err, kErrWaitMma)) {
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
              tc_mma_f16_pair(d_tmem, ad, bd, idesc, (kb | ks) != 0 ? 1u : 0u);
            }
            tc_commit_pair(empty_bar(stage), 0x3);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          tc_commit_pair(accf_bar(acc), 0x3);
          acc ^= 1u;
          if (acc == 0) acc_phase ^= 1u;
        }
        // All MMAs issued by this thread are complete once this commit arrives.
        tc_commit_pair(mma_done_bar, 0x1);
        mbar_wait(mma_done_bar, 0, err, kErrWaitMma);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const uint32_t q = warp & 3u;   // TMEM lane quarter this warp may access
    const uint32_t ew = warp - 2u;  // staging-buffer owner index
    uint8_t* out_buf0 = gbase + kOffOut + ew * 2u * kOutBufBytes;
    const uint32_t out_addr0 = base + kOffOut + ew * 2u * kOutBufBytes;
    uint32_t acc = 0, acc_phase = 0, ob = 0;
    for (int t = pair; t < num_tiles; t += num_pairs) {
      int mb, nb;
      pair_tile_coords(t, num_m, num_n, mb, nb);
      if (!mbar_wait_cluster(accf_bar(acc), acc_phase, err, kErrWaitEpilogue)) break;
      tc_fence_after_sync();
      const int row0 = mb * PM + static_cast<int>(rank) * HM + 32 * static_cast<int>(q);
      const int nslices = min(PN / 64, (N - nb * PN + 63) / 64);  // slices with columns inside Y
#pragma unroll 1
      for (int c = 0; c < nslices; ++c) {
        uint32_t r[64];
        const uint32_t taddr = tmem_base + ((32u * q) << 16) + acc * PN + c * 64;
        tmem_ld_32x32b_x32(taddr, r);
        tmem_ld_32x32b_x32(taddr + 32, r + 32);
        tmem_ld_wait();
        if (c == nslices - 1) {
          // This warp has read its whole share of the accumulator: hand it
          // back to the even CTA's MMA issuer.
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(acce_bar(acc), 0));
        }
        // The TMA store issued from this buffer two slices ago must have read it.
        if (lane == 0) bulk_wait_group_read<1>();
        __syncwarp();
        uint8_t* buf = out_buf0 + ob * kOutBufBytes;
        const int n0 = nb * PN + c * 64;
        switch (act) {
          case kActRelu:
            tcgemm::epilogue_slice<kBF16, kActRelu>(r, bias, n0, N, buf, lane);
            break;
          case kActGeluErf:
            tcgemm::epilogue_slice<kBF16, kActGeluErf>(r, bias, n0, N, buf, lane);
            break;
          case kActSoftplus:
            tcgemm::epilogue_slice<kBF16, kActSoftplus>(r, bias, n0, N, buf, lane);
            break;
          default:
            tcgemm::epilogue_slice<kBF16, kActNone>(r, bias, n0, N, buf, lane);
            break;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && row0 < M) {  // rows beyond Y (a ragged last pair row) are not stored
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

  // Neither CTA leaves (or frees the pair's TMEM) while the pair's MMAs may
  // still read its shared memory: the even CTA has waited for all of them.
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

}  // namespace tcpair

bool gemm_tc_pair_supported(int64_t M, int64_t N, int64_t K) { return M >= 1 && N >= 1 && K >= 1; }

cudaError_t launch_gemm_tc_pair(const DeviceCtx& dev, bool bf16, int64_t M, int64_t N, int64_t K, const void* A,
                                const void* B, const void* bias, void* Y, int act, cudaStream_t stream) {
  using namespace tcpair;
  if (!gemm_tc_pair_supported(M, N, K)) return cudaErrorNotSupported;
  const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap ta, tb, ty;
  cudaError_t e;
  if ((e = encode_tmap_2d(&ta, dt, 2, A, M, K, HM, BK, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess) return e;
  if ((e = encode_tmap_2d(&tb, dt, 2, B, K, N, BK, 64, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess) return e;
  if ((e = encode_tmap_2d(&ty, dt, 2, Y, M, N, 32, 64, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess) return e;

  auto kernel = bf16 ? gemm_bias_act_tc_pair_kernel<true> : gemm_bias_act_tc_pair_kernel<false>;
  if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes)) != cudaSuccess)
    return e;
  // One pair per two SMs, as many as can be resident at once (the kernel is
  // persistent: a pair that had to wait for another to finish would run its
  // tiles after everyone else).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(dev.sm_count & ~1));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  // Resident pairs per device and dtype, queried once (0: not yet known).
  static std::atomic<int> resident[64][2];
  const int di = dev.device >= 0 && dev.device < 64 ? dev.device : 0;
  int max_pairs = resident[di][bf16 ? 1 : 0].load(std::memory_order_relaxed);
  if (max_pairs == 0) {
    if ((e = cudaOccupancyMaxActiveClusters(&max_pairs, kernel, &cfg)) != cudaSuccess) return e;
    if (max_pairs < 1) return cudaErrorNotSupported;
    resident[di][bf16 ? 1 : 0].store(max_pairs, std::memory_order_relaxed);
  }
  const int64_t tiles = ((M + PM - 1) / PM) * ((N + PN - 1) / PN);
  const int pairs = static_cast<int>(tiles < max_pairs ? tiles : max_pairs);
  cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
  return cudaLaunchKernelEx(&cfg, kernel, ta, tb, ty, static_cast<const uint16_t*>(bias), static_cast<int>(M),
                            static_cast<int>(N), static_cast<int>(K), act, dev.err_word);
}

}  // namespace coalesce
