// fp32 GEMM with a fused bias + activation epilogue on the FP32 FMA pipe.
//
//   Y[M, N] = act(A[M, K] . B[K, N] + bias[N]),  fp32 products and sums.
//
// FP32-exact semantics are not a tensor-core contraction, so this path stays
// on FFMA, with register tiling (the "Coalesce" README, "Register tiling")
// sized for a GB300 SM: every thread keeps an 8 x 8 block of outputs in
// registers and, per k, combines 8 values of A with 8 values of B from shared
// memory into 64 FMAs.
//
//   * CTA tile 128 x 128, k-slab 32, 256 threads, an 8 x 8 patch per thread
//     (rows ty + 16 i, columns 4 tx + {0..3} and 64 + 4 tx + {0..3}):
//     per four k, 8 float4 loads of A (four k values of a row each) and 8 of
//     B feed 256 FMAs.
//   * Operands reach shared memory by TMA, A and B each as stored, through a
//     ring of six 32 KiB stages with full/empty mbarriers (bounded waits);
//     TMA zero-fills the ragged edges, and no CTA-wide barrier runs per slab.
//     A's 128-byte rows are 128-B swizzled by the TMA, so that the two rows a
//     warp reads at once fall in different banks.
//   * Blocked accumulation: each 32-deep slab is summed into a fresh fp32
//     partial that is then added to the running sum.  Plain sequential fp32
//     accumulation over K = 4096 of U(-1,1) products has an error of ~3e-5
//     (one sigma), too close to the 1e-4 tolerance; two-level summation
//     shrinks it several-fold for one extra FADD per 32 FMAs.
//   * Epilogue: + bias[n], activation in fp32, float4 stores (Y written once).
//   * Shapes with 128 x 128 tiles for between a quarter and a half of the SMs
//     split K over a cluster of two CTAs per tile (every SM gets a CTA of the
//     larger tile); fewer tiles than that use the small-shape kernel below
//     (64 x 64 tiles, K split over a cluster of up to four); with more than
//     half the SMs' worth the larger tile runs whole.
#include "epilogue.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace coalesce {
namespace f32gemm {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int BK = 16;   // the small-shape kernel's k slab
constexpr int BKB = 32;  // the 128 x 128 kernel's k slab
constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t f32_cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void f32_cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Read a float4 from the shared memory of CTA `rank` of this cluster.
__device__ __forceinline__ float4 ld_dsmem_f32x4(const float* local_ptr, uint32_t rank) {
  const uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(local_ptr));
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(remote)
               : "memory");
  return v;
}

// Tile order: groups of kGroupRows tile rows, column by column within a
// group (every other group walking its columns backwards, so that it starts
// on the B panels the previous group ended on), so that the CTAs resident at
// one time (one per SM) cover 16 tile rows x ~10 tile columns: their A and B
// panels (at 4096^3, 32 MB and ~19 MB) stay in L2 while the group is worked
// through, and each B panel is read from DRAM about once per group instead
// of once per wave.  The order changes which CTA computes a tile, never how:
// results are bit-identical to any other order.
constexpr int kGroupRows = 16;

__device__ __forceinline__ void f32_tile_coords(int tile, int num_m, int num_n, int& mb, int& nb) {
  const int per_group = kGroupRows * num_n;
  const int grp = tile / per_group;
  const int first = grp * kGroupRows;
  const int rows = min(kGroupRows, num_m - first);
  const int local = tile - grp * per_group;
  mb = first + local % rows;
  nb = local / rows;
  if (grp & 1) nb = num_n - 1 - nb;  // serpentine: a group starts on the B panels the previous one ended on
}

// Operand pipeline: each 32-deep k slab (A as stored, 128 rows x 32 k; B as
// stored, 32 k x 128 columns) is TMA-loaded into a ring of kStages
// shared-memory stages.  The warps wait for a stage's bytes on its `full`
// barrier and release it with one arrival each on its `empty` barrier.  Warp
// 0 issues the first kStages - 1 slabs; after that, warp j mod 8 (one lane)
// refills the stage of slab j - 1 with slab j + kStages - 1 once it has
// finished slab j, so it waits only for warps more than one slab behind it,
// and that wait is spread over all eight warps.  TMA zero-fills what lies
// beyond M, N or K.
constexpr int kStages = 6;
constexpr uint32_t kStageBytes = (BM * BKB + BKB * BN) * 4u;  // 32 KiB
constexpr int kComputeWarps = kThreads / 32;  // every warp computes and, in turn, issues the loads
constexpr int kF32Threads = kThreads;
constexpr uint32_t kF32SmemBytes = kStages * kStageBytes + 16u * kStages + 1024u;

// kSplitK = 2: a cluster of two CTAs shares each output tile, rank r summing
// the k slabs of the r-th half of K; rank 0 then adds rank 1's partial tile
// (read through distributed shared memory, in two halves that fit the
// operand stages) and runs the epilogue.  The order of the additions is
// fixed, so the result is deterministic.
//
// Thread (tx, ty) of the compute warps owns rows ty + 16 i (i < 8) and
// columns 4 tx + {0..3} and 64 + 4 tx + {0..3}.  A is read along k as float4
// (four k values of one row; the two rows a warp reads at once are adjacent,
// so they fall in different banks), B as two float4 per k.
template <int kAct, int kSplitK>
__global__ void __launch_bounds__(kF32Threads, 1)
    gemm_bias_act_f32_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                             const float* __restrict__ bias, float* __restrict__ Y, int M, int N, int K,
                             uint32_t* err) {
  extern __shared__ uint8_t f32_smem_raw[];
  // stages at a 1024-byte boundary (the 128-B swizzle pattern repeats every 1024 bytes), then the barriers
  const uint32_t raw = smem_u32(f32_smem_raw);
  const uint32_t sm0 = (raw + 1023u) & ~1023u;
  float* stages = reinterpret_cast<float*>(f32_smem_raw + (sm0 - raw));
  const uint32_t bar0 = sm0 + kStages * kStageBytes;
  auto full_bar = [&](int s) { return bar0 + 8u * static_cast<uint32_t>(s); };
  auto empty_bar = [&](int s) { return bar0 + 8u * static_cast<uint32_t>(kStages + s); };

  const int tid = threadIdx.x;
  const uint32_t warp = warp_index_uniform();
  const uint32_t lane = threadIdx.x % 32;
  const int num_n = (N + BN - 1) / BN;
  const int tile = static_cast<int>(blockIdx.x) / kSplitK;
  const uint32_t rank = kSplitK > 1 ? f32_cluster_ctarank() : 0u;
  int mb, nb;
  f32_tile_coords(tile, (M + BM - 1) / BM, num_n, mb, nb);
  const int m0 = mb * BM;
  const int n0 = nb * BN;

  const int num_kt_all = (K + BKB - 1) / BKB;
  // this CTA's k slabs: all of them, or one half of them per cluster rank
  const int kt0 = kSplitK > 1 ? static_cast<int>(rank) * ((num_kt_all + 1) / 2) : 0;
  const int num_kt = kSplitK > 1 ? min(num_kt_all, kt0 + (num_kt_all + 1) / 2) : num_kt_all;
  const int nslab = num_kt > kt0 ? num_kt - kt0 : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), kComputeWarps);
    }
    fence_mbarrier_init();
  }
  __syncthreads();

  const int tx = tid % 16;
  const int ty = tid / 16;
  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

  bool ok = true;
  // issue the loads of slab jn (one warp at a time; every lane of it calls)
  auto produce = [&](int jn) {
    const int sn = jn % kStages;
    if (jn >= kStages)
      ok = mbar_wait_warp(empty_bar(sn), static_cast<uint32_t>((jn / kStages) - 1) & 1u, err, kErrWaitF32);
    if (ok && lane == 0) {
      const int k0 = (kt0 + jn) * BKB;
      const uint32_t dst = sm0 + static_cast<uint32_t>(sn) * kStageBytes;
      mbar_arrive_expect_tx(full_bar(sn), kStageBytes);
      tma_load_2d(dst, &tma_a, full_bar(sn), k0, m0);
      tma_load_2d(dst + BM * BKB * 4u, &tma_b, full_bar(sn), n0, k0);
    }
    __syncwarp();
  };
  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tma_a);
      tma_prefetch_desc(&tma_b);
    }
    for (int jn = 0; jn < kStages - 1 && jn < nslab; ++jn) produce(jn);
  }
  for (int j = 0; ok && j < nslab; ++j) {
    const int s = j % kStages;
    if (!mbar_wait_warp(full_bar(s), static_cast<uint32_t>(j / kStages) & 1u, err, kErrWaitF32)) break;
    const float* As = stages + static_cast<size_t>(s) * (kStageBytes / 4);  // [BM][BKB], 128-B swizzled
    const float* Bs = As + BM * BKB;                                       // [BKB][BN]
    float part[8][8];
#pragma unroll
    for (int kq = 0; kq < BKB / 4; ++kq) {
      float4 af[8];
      // 16-byte chunk kq of row r sits at chunk kq ^ (r & 7); r & 7 = ty & 7 for every row of this thread
      const float* arow = As + ty * BKB + 4 * (kq ^ (ty & 7));
#pragma unroll
      for (int i = 0; i < 8; ++i) af[i] = *reinterpret_cast<const float4*>(arow + 16 * i * BKB);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int k = 4 * kq + kk;
        const float4 b0 = *reinterpret_cast<const float4*>(Bs + k * BN + tx * 4);
        const float4 b1 = *reinterpret_cast<const float4*>(Bs + k * BN + 64 + tx * 4);
        float a[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] = kk == 0 ? af[i].x : kk == 1 ? af[i].y : kk == 2 ? af[i].z : af[i].w;
        const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
        // columns outer, rows inner
#pragma unroll
        for (int jj = 0; jj < 8; ++jj)
#pragma unroll
          for (int i = 0; i < 8; ++i) part[i][jj] = (k == 0) ? a[i] * b[jj] : fmaf(a[i], b[jj], part[i][jj]);
      }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) acc[i][jj] += part[i][jj];
    __syncwarp();
    mbar_arrive_if(empty_bar(s), lane == 0 ? 1u : 0u);
    if (warp == static_cast<uint32_t>(j % kComputeWarps) && j + kStages - 1 < nslab) produce(j + kStages - 1);
  }
  // every stage has been read (and no load is in flight) before the stages
  // serve the split-K exchange
  __syncthreads();

  if constexpr (kSplitK > 1) {
    // Rank 1 publishes its partial tile in two halves (rows i < 4, then i >= 4)
    // through its operand stages; rank 0 adds each half to its own.
    // per half: columns 0..3 of each thread's four rows at the start of stage
    // 0, columns 4..7 at the start of stage 1 (4 x 256 threads x 4 floats =
    // 16 KiB each)
    float* red = stages;
    float* red2 = stages + kStageBytes / 4;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (rank == 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          *reinterpret_cast<float4*>(red + (i * kThreads + tid) * 4) =
              make_float4(acc[4 * h + i][0], acc[4 * h + i][1], acc[4 * h + i][2], acc[4 * h + i][3]);
          *reinterpret_cast<float4*>(red2 + (i * kThreads + tid) * 4) =
              make_float4(acc[4 * h + i][4], acc[4 * h + i][5], acc[4 * h + i][6], acc[4 * h + i][7]);
        }
      }
      f32_cluster_sync();
      if (rank == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 p = ld_dsmem_f32x4(red + (i * kThreads + tid) * 4, 1);
          const float4 q = ld_dsmem_f32x4(red2 + (i * kThreads + tid) * 4, 1);
          acc[4 * h + i][0] += p.x;
          acc[4 * h + i][1] += p.y;
          acc[4 * h + i][2] += p.z;
          acc[4 * h + i][3] += p.w;
          acc[4 * h + i][4] += q.x;
          acc[4 * h + i][5] += q.y;
          acc[4 * h + i][6] += q.z;
          acc[4 * h + i][7] += q.w;
        }
      }
      // rank 1's stages are reused (or freed) only after rank 0 has read them
      f32_cluster_sync();
    }
    if (rank != 0) return;
  }

  // Epilogue: bias + activation, float4 stores.
  const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
  float bv[8];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int gn = n0 + 64 * h + tx * 4;
    float4 b4 = zero4;
    if (bias != nullptr && gn < N) b4 = __ldg(reinterpret_cast<const float4*>(bias + gn));
    bv[4 * h + 0] = b4.x;
    bv[4 * h + 1] = b4.y;
    bv[4 * h + 2] = b4.z;
    bv[4 * h + 3] = b4.w;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int gm = m0 + ty + 16 * i;
    if (gm >= M) continue;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int gn = n0 + 64 * h + tx * 4;
      if (gn >= N) continue;
      float4 o;
      o.x = act_apply<kAct>(acc[i][4 * h + 0] + bv[4 * h + 0]);
      o.y = act_apply<kAct>(acc[i][4 * h + 1] + bv[4 * h + 1]);
      o.z = act_apply<kAct>(acc[i][4 * h + 2] + bv[4 * h + 2]);
      o.w = act_apply<kAct>(acc[i][4 * h + 3] + bv[4 * h + 3]);
      *reinterpret_cast<float4*>(Y + static_cast<size_t>(gm) * N + gn) = o;
    }
  }
}


// ---------------------------------------------------------------------------
// Small shapes: 64 x 64 tiles, split along K across a thread-block cluster.
//
// With 128 x 128 tiles a 512^3 problem has 16 CTAs for 152 SMs.  Here each
// output tile is computed by a cluster of kSplit CTAs, CTA r summing the k
// slabs r, r + kSplit, ... (two-level accumulation as above); the partial
// tiles are then added in rank order through distributed shared memory by
// the cluster's rank-0 CTA, which applies bias and activation and stores Y.
// No global scratch is used and the result is deterministic.
// ---------------------------------------------------------------------------
constexpr int SBM = 64;
constexpr int SBN = 64;
constexpr int kSmallThreads = 256;

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Read a float from the shared memory of CTA `rank` of this cluster.
__device__ __forceinline__ float ld_dsmem_f32(const float* local_ptr, uint32_t rank) {
  uint32_t local = static_cast<uint32_t>(__cvta_generic_to_shared(local_ptr));
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
  return v;
}

template <int kAct, int kSplit>
__global__ void __launch_bounds__(kSmallThreads)
    gemm_bias_act_f32_small_kernel(const float* __restrict__ A, const float* __restrict__ B,
                                   const float* __restrict__ bias, float* __restrict__ Y, int M, int N, int K) {
  __shared__ __align__(16) float As[2][BK][SBM];
  __shared__ __align__(16) float Bs[2][BK][SBN];
  __shared__ __align__(16) float red[SBM * SBN];  // this CTA's partial tile, read by rank 0

  const int tid = threadIdx.x;
  const int tx = tid % 16;
  const int ty = tid / 16;
  const int tile = static_cast<int>(blockIdx.x) / kSplit;
  const uint32_t rank = cluster_ctarank();
  const int num_n = (N + SBN - 1) / SBN;
  const int m0 = (tile / num_n) * SBM;
  const int n0 = (tile % num_n) * SBN;

  const int a_row = tid / 4, a_col = (tid % 4) * 4;    // 64 rows x 16 k: one float4 each
  const int b_row = tid / 16, b_col = (tid % 16) * 4;  // 16 k x 64 cols: one float4 each
  float4 ra, rb;
  const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
  auto fetch = [&](int k0) {
    const int gm = m0 + a_row, gk = k0 + a_col;
    ra = (gm < M && gk < K) ? __ldg(reinterpret_cast<const float4*>(A + static_cast<size_t>(gm) * K + gk)) : zero4;
    const int bk = k0 + b_row, gn = n0 + b_col;
    rb = (bk < K && gn < N) ? __ldg(reinterpret_cast<const float4*>(B + static_cast<size_t>(bk) * N + gn)) : zero4;
  };
  auto stash = [&](int buf) {
    As[buf][a_col + 0][a_row] = ra.x;
    As[buf][a_col + 1][a_row] = ra.y;
    As[buf][a_col + 2][a_row] = ra.z;
    As[buf][a_col + 3][a_row] = ra.w;
    *reinterpret_cast<float4*>(&Bs[buf][b_row][b_col]) = rb;
  };

  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

  const int num_kt = (K + BK - 1) / BK;
  int kt = static_cast<int>(rank);
  if (kt < num_kt) {
    fetch(kt * BK);
    stash(0);
  }
  __syncthreads();
  int cur = 0;
  for (; kt < num_kt; kt += kSplit) {
    const bool more = kt + kSplit < num_kt;
    if (more) fetch((kt + kSplit) * BK);
    float part[4][4];
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      const float4 a4 = *reinterpret_cast<const float4*>(&As[cur][k][ty * 4]);
      const float4 b4 = *reinterpret_cast<const float4*>(&Bs[cur][k][tx * 4]);
      const float a[4] = {a4.x, a4.y, a4.z, a4.w};
      const float b[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) part[i][j] = (k == 0) ? a[i] * b[j] : fmaf(a[i], b[j], part[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] += part[i][j];
    if (more) stash(cur ^ 1);
    __syncthreads();
    cur ^= 1;
  }

  // Partial tile to shared memory, then rank 0 adds the partials in rank order.
#pragma unroll
  for (int i = 0; i < 4; ++i)
    *reinterpret_cast<float4*>(&red[(ty * 4 + i) * SBN + tx * 4]) =
        make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
  cluster_sync_all();
  if (rank == 0) {
    float bv[4] = {0.f, 0.f, 0.f, 0.f};
    const int gn = n0 + tx * 4;
    if (bias != nullptr && gn < N) {
      const float4 b4 = __ldg(reinterpret_cast<const float4*>(bias + gn));
      bv[0] = b4.x;
      bv[1] = b4.y;
      bv[2] = b4.z;
      bv[3] = b4.w;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float sum[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) sum[j] = acc[i][j];
      for (uint32_t r = 1; r < static_cast<uint32_t>(kSplit); ++r) {
#pragma unroll
        for (int j = 0; j < 4; ++j) sum[j] += ld_dsmem_f32(&red[(ty * 4 + i) * SBN + tx * 4 + j], r);
      }
      const int gm = m0 + ty * 4 + i;
      if (gm < M && gn < N) {
        float4 o;
        o.x = act_apply<kAct>(sum[0] + bv[0]);
        o.y = act_apply<kAct>(sum[1] + bv[1]);
        o.z = act_apply<kAct>(sum[2] + bv[2]);
        o.w = act_apply<kAct>(sum[3] + bv[3]);
        *reinterpret_cast<float4*>(Y + static_cast<size_t>(gm) * N + gn) = o;
      }
    }
  }
  // Keep every CTA's partial alive until rank 0 has read it.
  cluster_sync_all();
}

template <int kAct, int kSplit>
cudaError_t launch_small(int64_t M, int64_t N, int64_t K, const float* A, const float* B, const float* bias, float* Y,
                         cudaStream_t stream) {
  const int64_t tiles = ((M + SBM - 1) / SBM) * ((N + SBN - 1) / SBN);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles * kSplit));
  cfg.blockDim = dim3(kSmallThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kSplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_bias_act_f32_small_kernel<kAct, kSplit>, A, B, bias, Y, static_cast<int>(M),
                            static_cast<int>(N), static_cast<int>(K));
}

template <int kAct>
cudaError_t launch_small_split(int split, int64_t M, int64_t N, int64_t K, const float* A, const float* B,
                               const float* bias, float* Y, cudaStream_t stream) {
  switch (split) {
    case 4:
      return launch_small<kAct, 4>(M, N, K, A, B, bias, Y, stream);
    case 2:
      return launch_small<kAct, 2>(M, N, K, A, B, bias, Y, stream);
    default:
      return launch_small<kAct, 1>(M, N, K, A, B, bias, Y, stream);
  }
}

template <int kAct, int kSplitK>
cudaError_t launch_big_split(int64_t tiles, const CUtensorMap& ta, const CUtensorMap& tb, const float* bias, float* Y,
                             int m, int n, int k, uint32_t* err, cudaStream_t stream) {
  auto kernel = gemm_bias_act_f32_kernel<kAct, kSplitK>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kF32SmemBytes));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(tiles * kSplitK));
  cfg.blockDim = dim3(kF32Threads);
  cfg.dynamicSmemBytes = kF32SmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kSplitK;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = kSplitK > 1 ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, ta, tb, bias, Y, m, n, k, err);
}

template <int kAct>
cudaError_t launch_big(int split, int64_t tiles, const float* A, const float* B, const float* bias, float* Y, int m,
                       int n, int k, uint32_t* err, cudaStream_t stream) {
  CUtensorMap ta, tb;
  cudaError_t e;
  if ((e = encode_tmap_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, A, static_cast<uint64_t>(m),
                          static_cast<uint64_t>(k), BM, BKB, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return e;
  if ((e = encode_tmap_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, B, static_cast<uint64_t>(k),
                          static_cast<uint64_t>(n), BKB, BN, CU_TENSOR_MAP_SWIZZLE_NONE)) != cudaSuccess)
    return e;
  if (split == 2) return launch_big_split<kAct, 2>(tiles, ta, tb, bias, Y, m, n, k, err, stream);
  return launch_big_split<kAct, 1>(tiles, ta, tb, bias, Y, m, n, k, err, stream);
}

}  // namespace f32gemm

cudaError_t launch_gemm_f32(const DeviceCtx& dev, int64_t M, int64_t N, int64_t K, const float* A, const float* B,
                            const float* bias, float* Y, int act, cudaStream_t stream) {
  using namespace f32gemm;
  const int64_t tiles = ((N + BN - 1) / BN) * ((M + BM - 1) / BM);
  if (tiles > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  // Between a quarter and a half of the SMs' worth of 128 x 128 tiles: K
  // split over a cluster of two CTAs per tile, so that every SM gets a CTA
  // of the larger tile.  The choice depends on the SM count, and with it the
  // order of the fp32 sums: results are bit-reproducible on one device model,
  // not across models with other SM counts (within tolerance on every one).
  const int split = (2 * tiles <= dev.sm_count && 4 * tiles >= dev.sm_count && K >= 2 * BKB) ? 2 : 1;
  if (2 * tiles <= dev.sm_count && split == 1) {
    // 128 x 128 tiles would leave most SMs idle: 64 x 64 tiles, and K split
    // over a cluster of up to four CTAs while the CTAs still fit one per SM
    // (and each keeps at least one 16-deep k slab).  Measured at N = M = K:
    // 256 and 512 run fastest with splits of 4 and 2 (15 and 27 us; 25 and
    // 46 us with 8, whose rank-0 reduction of eight partials costs more than
    // the extra CTAs save), 1024 without a split.
    const int64_t small_tiles = ((N + SBN - 1) / SBN) * ((M + SBM - 1) / SBM);
    const int64_t kslabs = (K + BK - 1) / BK;
    int split = 1;
    while (split < 4 && small_tiles * split * 2 <= dev.sm_count && 2 * split <= kslabs) split *= 2;
    switch (act) {
      case kActRelu:
        return launch_small_split<kActRelu>(split, M, N, K, A, B, bias, Y, stream);
      case kActGeluErf:
        return launch_small_split<kActGeluErf>(split, M, N, K, A, B, bias, Y, stream);
      case kActSoftplus:
        return launch_small_split<kActSoftplus>(split, M, N, K, A, B, bias, Y, stream);
      default:
        return launch_small_split<kActNone>(split, M, N, K, A, B, bias, Y, stream);
    }
  }
  const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
  switch (act) {
    case kActRelu:
      return launch_big<kActRelu>(split, tiles, A, B, bias, Y, m, n, k, dev.err_word, stream);
    case kActGeluErf:
      return launch_big<kActGeluErf>(split, tiles, A, B, bias, Y, m, n, k, dev.err_word, stream);
    case kActSoftplus:
      return launch_big<kActSoftplus>(split, tiles, A, B, bias, Y, m, n, k, dev.err_word, stream);
    default:
      return launch_big<kActNone>(split, tiles, A, B, bias, Y, m, n, k, dev.err_word, stream);
  }
}

}  // namespace coalesce
