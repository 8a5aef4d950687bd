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
//     TMEM.  Row tiles of 128 rows live in a ring of S >= E + 1 shared-memory
//     slots of 128 x max(D, H) fp16: local tile i uses slot i mod S and is
//     processed by worker i mod E.  A worker runs its tile through every
//     layer: its leader thread issues the layer's MMAs (M = 128, N = H,
//     K = 16 steps) from the slot into TMEM; the four warps read the
//     accumulator back (tcgen05.ld, one TMEM lane = one row), round it to
//     fp16, apply the activation and write the result over the same slot in
//     the K-major swizzled layout the next layer's MMA reads.  The last
//     layer's fp16 result is TMA-stored from the slot.  Between layers
//     nothing leaves the SM.
//   * No producer warp: whoever frees a slot (its output store has been read)
//     refills it by TMA with the tile due there next (tile i + S), so loads of
//     later tiles, tensor-core work, epilogue math and stores of different
//     tiles overlap.
//   * The bias never costs an epilogue instruction: as soon as a warp has
//     read its accumulator columns it writes the NEXT layer's bias (fp32)
//     into them with tcgen05.st, and the next MMA accumulates on top of it.
//   * Softplus runs on packed fp16 pairs (one ex2.approx.f16x2 plus a short
//     polynomial, about four instructions per value), because the epilogue,
//     not the tensor core, sets the pace of a 64- or 128-wide chain.
// Ragged row tails are handled by TMA (zero-filled loads, clipped stores).
#include "epilogue.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace coalesce {
namespace mlp {

constexpr int BM = 128;
constexpr int kMaxLayers = 8;
constexpr int kMaxWorkers = 4;  // 16 warps: 4 per SM sub-partition, up to 128 registers each
constexpr int kMaxSlots = 8;
constexpr uint32_t kSmemLimit = 232448;  // opt-in maximum dynamic shared memory per block on sm_103a
constexpr uint32_t kWeightBudget = 160u * 1024u;

// Shared-memory plan, identical on host and device.  Small items (barriers,
// TMEM address, fp32 biases) sit at the start of the dynamic window; the
// swizzled operand buffers start at the next 1 KiB boundary after them.
struct Layout {
  // relative to the start of dynamic shared memory
  uint32_t bar_off;        // w_full, x_full[S], mma_done[E]
  uint32_t tmem_slot_off;
  uint32_t bias_off;
  uint32_t small_bytes;
  // relative to the 1 KiB-aligned big base
  uint32_t w_off[kMaxLayers];
  uint32_t slot_off;       // slot s at slot_off + s * slot_bytes
  uint32_t slots;          // S
  uint32_t slot_bytes;
  uint32_t big_bytes;
  uint32_t alloc_bytes;    // small + worst-case alignment padding + big
  uint32_t tmem_cols;      // allocated TMEM columns (power of two)
};

__host__ __device__ inline uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

__host__ __device__ inline Layout make_layout(int D, int H, int L, int E, int S) {
  Layout lo{};
  uint32_t off = 0;
  lo.bar_off = off;
  off += 8u * (1u + static_cast<uint32_t>(S + E));
  lo.tmem_slot_off = off;
  off += 16;
  lo.bias_off = align_up(off, 16);  // read as float4
  off = lo.bias_off + static_cast<uint32_t>(L * H) * 4u;
  lo.small_bytes = align_up(off, 16);
  uint32_t big = 0;
  for (int l = 0; l < L; ++l) {
    const uint32_t K = l == 0 ? D : H;
    lo.w_off[l] = big;
    big += static_cast<uint32_t>(H / 64) * K * 128u;
  }
  const int kmax = D > H ? D : H;
  lo.slot_bytes = static_cast<uint32_t>(kmax / 64) * BM * 128u;
  lo.slot_off = big;
  lo.slots = static_cast<uint32_t>(S);
  big += static_cast<uint32_t>(S) * lo.slot_bytes;
  lo.big_bytes = big;
  // dynamic shared memory is at least 16-byte aligned: at most 1008 bytes of padding
  lo.alloc_bytes = lo.small_bytes + 1008u + big;
  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>(E * H)) cols <<= 1;
  lo.tmem_cols = cols;
  return lo;
}

struct Params {
  CUtensorMap x_map;                  // x [rows, D], box 128 x 64, 128-B swizzle
  CUtensorMap out_map;                // out [rows, H], box 32 x 64, 128-B swizzle
  CUtensorMap w_map[kMaxLayers];      // W_l [K_l, H], box K_l x 64, 128-B swizzle
  const uint16_t* bias[kMaxLayers];   // b_l[H] fp16, or nullptr
  Layout lo;                          // shared-memory plan (host-computed)
  int rows, D, H, L, act, workers;
  uint32_t* err;
};

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// 64 accumulator columns of one row (fp32 bits in r) -> fp16 -> activation,
// written to row `row` of column block `cb` of the K-major 128-B-swizzled slot
// (16-byte chunk j of a row lives at chunk j ^ (row & 7)).
template <int kAct>
__device__ __forceinline__ void epilogue_block64(const uint32_t* r, uint8_t* slot, int cb, uint32_t row) {
  uint8_t* rowp = slot + static_cast<uint32_t>(cb) * (BM * 128u) + row * 128u;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float lo = __uint_as_float(r[8 * j + 2 * k]);
      const float hi = __uint_as_float(r[8 * j + 2 * k + 1]);
      if constexpr (kAct == kActSoftplus) {
        w[k] = softplus_f16x2(pack_f16x2(lo, hi));
      } else if constexpr (kAct == kActNone) {
        w[k] = pack_f16x2(lo, hi);
      } else {
        w[k] = pack_f16x2(act_apply<kAct>(lo), act_apply<kAct>(hi));
      }
    }
    const uint32_t phys = static_cast<uint32_t>(j) ^ (row & 7u);
    *reinterpret_cast<uint4*>(rowp + phys * 16u) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Write bias[c0 .. c0+63] (fp32, shared memory) into this warp's 32 TMEM lanes,
// columns c0 .. c0+63 of its accumulator, so that the next MMA adds onto it.
__device__ __forceinline__ void preload_bias64(uint32_t tmem_row, const float* bias_s, int c0) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t b[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 v = *reinterpret_cast<const float4*>(bias_s + c0 + 32 * h + 4 * i);
      b[4 * i] = __float_as_uint(v.x);
      b[4 * i + 1] = __float_as_uint(v.y);
      b[4 * i + 2] = __float_as_uint(v.z);
      b[4 * i + 3] = __float_as_uint(v.w);
    }
    tmem_st_32x32b_x32(tmem_row + static_cast<uint32_t>(c0 + 32 * h), b);
  }
}

template <int kAct>
__global__ void __launch_bounds__(128 * kMaxWorkers, 1) mlp_fused_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ int bias_nonzero[kMaxLayers];
  const int E = p.workers;
  const Layout& lo = p.lo;
  const int S = static_cast<int>(lo.slots);
  const uint32_t sbase = smem_u32(smem_raw);                        // small items
  const uint32_t base = (sbase + lo.small_bytes + 1023u) & ~1023u;  // swizzled buffers
  uint8_t* gbase = smem_raw + (base - sbase);
  const uint32_t warp = threadIdx.x / 32;
  const uint32_t lane = threadIdx.x % 32;
  const int num_tiles = (p.rows + BM - 1) / BM;
  // tiles of this CTA: blockIdx.x + i * gridDim.x, i = 0 .. my_tiles - 1
  const int my_tiles = blockIdx.x < num_tiles ? (num_tiles - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;

  const uint32_t w_full = sbase + lo.bar_off;
  auto x_full = [&](int slot) { return sbase + lo.bar_off + 8u * (1 + slot); };
  auto mma_done = [&](int g) { return sbase + lo.bar_off + 8u * (1 + S + g); };
  auto slot_addr = [&](int slot) { return lo.slot_off + static_cast<uint32_t>(slot) * lo.slot_bytes; };
  const uint32_t xbytes = static_cast<uint32_t>(p.D) * BM * 2u;
  // TMA load of local tile i into its slot (one 64-column box per column block).
  auto load_tile = [&](int i) {
    const int slot = i % S;
    const int t = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
    mbar_arrive_expect_tx(x_full(slot), xbytes);
    for (int c = 0; c < p.D / 64; ++c)
      tma_load_2d(base + slot_addr(slot) + static_cast<uint32_t>(c) * BM * 128u, &p.x_map, x_full(slot), c * 64,
                  t * BM);
  };

  // ---- set-up: barriers, TMEM, biases (fp32), weights and the first S tiles (TMA)
  if (threadIdx.x == 0) {
    mbar_init(w_full, 1);
    for (int i = 0; i < S; ++i) mbar_init(x_full(i), 1);
    for (int g = 0; g < E; ++g) mbar_init(mma_done(g), 1);
    fence_mbarrier_init();
  }
  if (warp == 0) {
    tmem_alloc(sbase + lo.tmem_slot_off, lo.tmem_cols);
    tmem_relinquish_alloc_permit();
  }
  float* bias_s = reinterpret_cast<float*>(smem_raw + lo.bias_off);
  if (threadIdx.x < kMaxLayers) bias_nonzero[threadIdx.x] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < p.L * p.H; i += blockDim.x) {
    const int l = i / p.H, n = i % p.H;
    const float v = p.bias[l] != nullptr ? __half2float(__ushort_as_half(p.bias[l][n])) : 0.0f;
    bias_s[i] = v;
    if (v != 0.0f) bias_nonzero[l] = 1;  // benign race: every writer stores 1
  }
  if (threadIdx.x == 0) {
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
    for (int i = 0; i < S && i < my_tiles; ++i) load_tile(i);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem_raw + lo.tmem_slot_off);

  // ------------------------------------------------------------ row-tile workers
  const int g = static_cast<int>(warp) / 4;
  const uint32_t q = warp & 3u;               // TMEM lane quarter of this warp
  const uint32_t row = 32u * q + lane;        // row within the tile (= TMEM lane)
  const bool leader = q == 0 && lane == 0;
  const uint32_t tmem_acc = tmem_base + static_cast<uint32_t>(g * p.H);
  const uint32_t tmem_row = tmem_acc + ((32u * q) << 16);
  const uint32_t bar_id = 1u + static_cast<uint32_t>(g);
  const int nblk = p.H / 64;
  uint32_t mma_phase = 0;
  // The first MMA of the first tile accumulates onto b_0.
  if (bias_nonzero[0]) {
    for (int cb = 0; cb < nblk; ++cb) preload_bias64(tmem_row, bias_s, 64 * cb);
    tmem_st_wait();
  }
  tc_fence_before_sync();
  named_bar_sync(bar_id, 128);
  bool ok = mbar_wait(w_full, 0, p.err, kErrWaitMlp);
  int prev = -1;  // this worker's previous tile: its slot is refilled once its store has been read
  for (int i = g; ok && i < my_tiles; i += E) {
    const int slot = i % S;
    const int t = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
    if (!mbar_wait(x_full(slot), (i / S) & 1, p.err, kErrWaitMlp)) {
      ok = false;
      break;
    }
    uint8_t* sl = gbase + slot_addr(slot);
    const uint32_t slot_a = base + slot_addr(slot);
    for (int l = 0; l < p.L; ++l) {
      const int K = l == 0 ? p.D : p.H;
      if (leader) {
        tc_fence_after_sync();
        const uint32_t idesc = idesc_f16_f32acc(false, false, true, BM, static_cast<uint32_t>(p.H));
        const uint32_t wa = base + lo.w_off[l];
        const uint32_t acc0 = bias_nonzero[l] ? 1u : 0u;
        for (int ks = 0; ks < K / 16; ++ks) {
          const uint64_t ad =
              smem_desc_sw128(slot_a + static_cast<uint32_t>(ks / 4) * BM * 128u + (ks % 4) * 32u, 16, 1024);
          const uint64_t bd =
              smem_desc_sw128(wa + static_cast<uint32_t>(ks) * 2048u, static_cast<uint32_t>(K) * 128u, 1024);
          tc_mma_f16(tmem_acc, ad, bd, idesc, ks > 0 ? 1u : acc0);
        }
        tc_commit(mma_done(g));
      }
      if (!mbar_wait(mma_done(g), mma_phase, p.err, kErrWaitMlp)) {
        ok = false;
        break;
      }
      mma_phase ^= 1u;
      tc_fence_after_sync();
      const bool last = (l == p.L - 1);
      const int next_l = last ? 0 : l + 1;  // the next MMA on this accumulator
      const bool pre = bias_nonzero[next_l] != 0;
      const float* bnext = bias_s + next_l * p.H;
      for (int cb = 0; cb < nblk; ++cb) {
        uint32_t r[64];
        tmem_ld_32x32b_x32(tmem_row + static_cast<uint32_t>(64 * cb), r);
        tmem_ld_32x32b_x32(tmem_row + static_cast<uint32_t>(64 * cb + 32), r + 32);
        tmem_ld_wait();
        if (last) {
          epilogue_block64<kActNone>(r, sl, cb, row);
        } else {
          epilogue_block64<kAct>(r, sl, cb, row);
        }
        // These accumulator columns have been read: seed them with the next bias.
        if (pre) preload_bias64(tmem_row, bnext, 64 * cb);
      }
      if (l == 0 && prev >= 0 && lane == 0) bulk_wait_group_read<0>();  // previous tile's store has read its slot
      // TMEM reads (and bias writes) done, slot rewritten: publish to the tensor core / TMA.
      if (pre) tmem_st_wait();
      tc_fence_before_sync();
      fence_proxy_async_smem();
      named_bar_sync(bar_id, 128);
      if (l == 0 && prev >= 0) {
        // All four warps' stores from the previous tile's slot are done: refill it.
        if (leader && prev + S < my_tiles) load_tile(prev + S);
        prev = -1;
      }
    }
    if (!ok) break;
    // This warp's 32 rows of the finished tile go out by TMA.
    if (lane == 0) {
      for (int c = 0; c < nblk; ++c)
        tma_store_2d(&p.out_map, slot_a + static_cast<uint32_t>(c) * BM * 128u + 32u * q * 128u, c * 64,
                     t * BM + static_cast<int>(32u * q));
      bulk_commit_group();
    }
    prev = i;
  }
  if (lane == 0) bulk_wait_group<0>();
  __syncwarp();
  // A refill this worker still owes (its last tile's slot) is never needed: no later tile uses it.

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
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
  // Most row-tile workers that fit TMEM and shared memory with a ring of at
  // least E + 1 slots (one tile in flight per worker plus one being loaded).
  int E = 0, S = 0;
  for (int e = kMaxWorkers; e >= 1 && E == 0; --e) {
    if (e * H > 512) continue;
    for (int sl = kMaxSlots; sl >= e + 1; --sl) {
      if (make_layout(D, H, L, e, sl).alloc_bytes <= kSmemLimit) {
        E = e;
        S = sl < 2 * e ? sl : 2 * e;
        break;
      }
    }
  }
  if (E == 0) return cudaErrorNotSupported;
  const Layout lo = make_layout(D, H, L, E, S);
  const uint32_t smem = lo.alloc_bytes;
  if (lo.bias_off % 16 != 0 || lo.small_bytes % 16 != 0) return cudaErrorNotSupported;

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
  p.lo = lo;
  p.err = dev.err_word;

  void (*kernel)(Params);
  switch (act) {
    case kActSoftplus:
      kernel = mlp_fused_kernel<kActSoftplus>;
      break;
    case kActRelu:
      kernel = mlp_fused_kernel<kActRelu>;
      break;
    case kActGeluErf:
      kernel = mlp_fused_kernel<kActGeluErf>;
      break;
    default:
      kernel = mlp_fused_kernel<kActNone>;
      break;
  }
  if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
    return e;
  const int64_t tiles = (rows + BM - 1) / BM;
  const int grid = static_cast<int>(tiles < dev.sm_count ? tiles : dev.sm_count);
  kernel<<<grid, 128 * E, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace coalesce
