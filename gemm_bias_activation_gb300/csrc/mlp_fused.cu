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
//   * Row tiles of 128 rows live in a ring of S shared-memory slots of
//     128 x max(D, H) fp16; CTA-local tile i uses slot i mod S.  V = E * P row
//     tiles are in flight at once: E "workers" of 4 warps each interleave P
//     tiles, and virtual worker v (worker v / P, lane v mod P) owns TMEM
//     columns [v H, v H + H) and the tiles v, v + V, v + 2V, ...
//   * Whoever finishes last issues the next step, so no warp waits for a
//     dedicated issuer: the last of a worker's four warps to finish a stage's
//     epilogue (a shared-memory acq_rel counter per virtual worker) issues the
//     next layer's MMAs (M = 128, N = H, K = 16 steps) and commits them to
//     mma_done[v]; the last warp to release a slot (its output store has read
//     it) refills it by TMA with the tile due there next and prefetches a tile
//     further ahead into L2, so HBM latency stays off the critical path.
//   * The epilogue warps of a worker go stage by stage (round, layer, lane):
//     wait for mma_done, read the accumulator back (tcgen05.ld, one TMEM lane
//     = one row), round it to fp16, apply the activation and write the
//     result over the tile's slot in the K-major swizzled layout the next
//     layer's MMA reads; after the last layer each warp TMA-stores its own 32
//     rows.  Between layers nothing leaves the SM.  Warps never wait for each
//     other directly: only for mbarriers (MMA completion, landed tiles).
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
constexpr int kMaxWorkers = 4;                       // epilogue warpgroups
constexpr int kMaxVirtual = 8;                       // row tiles in flight
constexpr int kMaxSlots = 12;
constexpr int kThreads = 128 * kMaxWorkers;
constexpr int kPrefetchAhead = 4;                    // tiles prefetched into L2 beyond the ring
constexpr uint32_t kSmemLimit = 232448;              // opt-in maximum dynamic shared memory per block
constexpr uint32_t kWeightBudget = 160u * 1024u;

// Shared-memory plan, identical on host and device.  Small items (barriers,
// TMEM address, fp32 biases) sit at the start of the dynamic window; the
// swizzled operand buffers start at the next 1 KiB boundary after them.
struct Layout {
  // relative to the start of dynamic shared memory
  uint32_t bar_off;        // w_full, x_full[S], mma_done[V], then counters:
                           // ready_cnt[V] (warps done with v's current stage),
                           // free_cnt[S] (warps whose store has read slot s)
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

// V row tiles in flight (V accumulators), S slots.
__host__ __device__ inline Layout make_layout(int D, int H, int L, int V, int S) {
  Layout lo{};
  uint32_t off = 0;
  lo.bar_off = off;
  off += 8u * (1u + static_cast<uint32_t>(S + V)) + 4u * static_cast<uint32_t>(V + S);
  off = align_up(off, 8);
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
  while (cols < static_cast<uint32_t>(V * H)) cols <<= 1;
  lo.tmem_cols = cols;
  return lo;
}

struct Params {
  CUtensorMap x_map;                  // x [rows, D], box 128 x 64, 128-B swizzle
  CUtensorMap out_map;                // out [rows, H], box 32 x 64, 128-B swizzle
  CUtensorMap w_map[kMaxLayers];      // W_l [K_l, H], box K_l x 64, 128-B swizzle
  const uint16_t* bias[kMaxLayers];   // b_l[H] fp16, or nullptr
  Layout lo;                          // shared-memory plan (host-computed)
  int rows, D, H, L;
  int workers;                        // E
  int pp;                             // P: row tiles in flight per worker
  uint32_t* err;
};

// 64 accumulator columns of one row (fp32 bits in r) -> fp16 -> activation,
// written to the row `rowp` of a 128-B-swizzled column block (16-byte chunk j
// of a row lives at chunk j ^ (row & 7)).
template <int kAct>
__device__ __forceinline__ void epilogue_row64(const uint32_t* r, uint8_t* rowp, uint32_t row_sw) {
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
    *reinterpret_cast<uint4*>(rowp + ((static_cast<uint32_t>(j) ^ row_sw) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Write bias[c0 .. c0+31] (fp32, shared memory) into this warp's 32 TMEM lanes,
// columns c0 .. c0+31 of its accumulator, so that the next MMA adds onto it.
__device__ __forceinline__ void preload_bias32(uint32_t tmem_row, const float* bias_s, int c0) {
  uint32_t b[32];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 v = *reinterpret_cast<const float4*>(bias_s + c0 + 4 * i);
    b[4 * i] = __float_as_uint(v.x);
    b[4 * i + 1] = __float_as_uint(v.y);
    b[4 * i + 2] = __float_as_uint(v.z);
    b[4 * i + 3] = __float_as_uint(v.w);
  }
  tmem_st_32x32b_x32(tmem_row + static_cast<uint32_t>(c0), b);
}

template <int kAct>
__global__ void __launch_bounds__(kThreads, 1) mlp_fused_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ int bias_nonzero[kMaxLayers];
  const int E = p.workers;
  const int P = p.pp;
  const int V = E * P;
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
  auto x_full = [&](int s) { return sbase + lo.bar_off + 8u * (1 + s); };
  auto mma_done = [&](int v) { return sbase + lo.bar_off + 8u * (1 + S + v); };
  const uint32_t cnt_base = sbase + lo.bar_off + 8u * (1 + S + V);
  auto ready_cnt = [&](int v) { return cnt_base + 4u * v; };
  auto free_cnt = [&](int s) { return cnt_base + 4u * (V + s); };
  auto slot_addr = [&](int s) { return lo.slot_off + static_cast<uint32_t>(s) * lo.slot_bytes; };
  auto tile_row = [&](int i) { return (static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x)) * BM; };
  const uint32_t xbytes = static_cast<uint32_t>(p.D) * BM * 2u;
  auto prefetch_tile = [&](int i) {
    for (int c = 0; c < p.D / 64; ++c) tma_prefetch_l2_2d(&p.x_map, c * 64, tile_row(i));
  };

  // ---- set-up: barriers, counters, TMEM, biases (fp32), weights and the first S tiles (TMA)
  if (threadIdx.x == 0) {
    mbar_init(w_full, 1);
    for (int s = 0; s < S; ++s) mbar_init(x_full(s), 1);
    for (int v = 0; v < V; ++v) mbar_init(mma_done(v), 1);
    fence_mbarrier_init();
  }
  for (int c = threadIdx.x; c < V + S; c += blockDim.x) reinterpret_cast<uint32_t*>(smem_raw + (cnt_base - sbase))[c] = 0;
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
    for (int i = 0; i < S && i < my_tiles; ++i) {  // tile i -> slot i, first load of each slot
      mbar_arrive_expect_tx(x_full(i), xbytes);
      for (int c = 0; c < p.D / 64; ++c)
        tma_load_2d(base + slot_addr(i) + static_cast<uint32_t>(c) * BM * 128u, &p.x_map, x_full(i), c * 64,
                    tile_row(i));
    }
    for (int i = S; i < S + kPrefetchAhead && i < my_tiles; ++i) prefetch_tile(i);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem_raw + lo.tmem_slot_off);

  const uint32_t idesc = idesc_f16_f32acc(false, false, true, BM, static_cast<uint32_t>(p.H));
  // Issue (no commit) layer l's MMAs for the tile in slot `slot` into
  // accumulator `acc_idx` (one thread).
  auto issue_mmas = [&](int acc_idx, int slot, int l) {
    const int K = l == 0 ? p.D : p.H;
    const uint32_t slot_a = base + slot_addr(slot);
    const uint32_t wa = base + lo.w_off[l];
    const uint32_t acc0 = bias_nonzero[l] ? 1u : 0u;
    const uint32_t d = tmem_base + static_cast<uint32_t>(acc_idx * p.H);
    for (int ks = 0; ks < K / 16; ++ks) {
      const uint64_t ad =
          smem_desc_sw128(slot_a + static_cast<uint32_t>(ks / 4) * BM * 128u + (ks % 4) * 32u, 16, 1024);
      const uint64_t bd =
          smem_desc_sw128(wa + static_cast<uint32_t>(ks) * 2048u, static_cast<uint32_t>(K) * 128u, 1024);
      tc_mma_f16(d, ad, bd, idesc, ks > 0 ? 1u : acc0);
    }
  };

  // ------------------------------------------------------------ row-tile workers
  // Worker g processes its row tiles in groups of P (tiles g P + a + m V for
  // a < P), all P tiles of a group together: one wait, one pass of fences and
  // one commit per layer for P x 128 rows.
  const int g = static_cast<int>(warp) / 4;
  const uint32_t q = warp & 3u;               // TMEM lane quarter of this warp
  const uint32_t row = 32u * q + lane;        // row within the tile (= TMEM lane)
  const uint32_t row_off = row * 128u;
  const uint32_t row_sw = row & 7u;
  const int ncols = p.H;
  bool ok = __all_sync(0xffffffffu, mbar_wait(w_full, 0, p.err, kErrWaitMlp));
  // Every accumulator starts out holding b_0 for its first MMA.
  if (bias_nonzero[0]) {
#pragma unroll
    for (int a = 0; a < 2; ++a) {
      if (a >= P) break;
      const uint32_t tmem_row = tmem_base + static_cast<uint32_t>((g * P + a) * p.H) + ((32u * q) << 16);
      for (int c0 = 0; c0 < ncols; c0 += 32) preload_bias32(tmem_row, bias_s, c0);
    }
    tmem_st_wait();
  }
  tc_fence_before_sync();
  __syncwarp();
  // Slot and load parity of each tile of the current group, advanced without
  // division: tile i + V sits V slots further on, wrapping at most once (V < S).
  int gs[2], gp[2];
#pragma unroll
  for (int a = 0; a < 2; ++a) {
    gs[a] = g * P + a;  // tile v < V < S lives in slot v, first load
    gp[a] = 0;
  }
  {
    const int first = g * P;
    const int na = my_tiles - first < P ? my_tiles - first : P;
    // The last warp of the worker to get here issues the first group's layer 0.
    if (lane == 0 && smem_atomic_add_acq_rel(ready_cnt(g), 1) % 4 == 3 && na > 0 && ok) {
      tc_fence_after_sync();
#pragma unroll
      for (int a = 0; a < 2; ++a) {
        if (a >= na) break;
        ok = ok && mbar_wait(x_full(gs[a]), 0u, p.err, kErrWaitMlp);
        if (ok) issue_mmas(g * P + a, gs[a], 0);
      }
      tc_commit(mma_done(g));
    }
  }
  ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  int pend_slot[2], pend_tile[2], npend = 0;  // slots this warp stored from, to release next stage
  for (int m = 0; ok; ++m) {
    const int first = g * P + m * V;
    if (first >= my_tiles) break;
    const int na = my_tiles - first < P ? my_tiles - first : P;
    for (int l = 0; l < p.L && ok; ++l) {
      const int k = m * p.L + l;  // stage count of this worker
      const bool got = mbar_wait(mma_done(g), k & 1, p.err, kErrWaitMlp);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const bool last = (l == p.L - 1);
      const int next_l = last ? 0 : l + 1;  // the next MMA on these accumulators
      const bool pre = bias_nonzero[next_l] != 0;
      const float* bnext = bias_s + next_l * p.H;
#pragma unroll
      for (int a = 0; a < 2; ++a) {
        if (a >= na) break;
        uint8_t* sl = gbase + slot_addr(gs[a]);
        const uint32_t tmem_row = tmem_base + static_cast<uint32_t>((g * P + a) * p.H) + ((32u * q) << 16);
        for (int c0 = 0; c0 < ncols; c0 += 64) {
          uint32_t acc[64];
          tmem_ld_32x32b_x32(tmem_row + static_cast<uint32_t>(c0), acc);
          tmem_ld_32x32b_x32(tmem_row + static_cast<uint32_t>(c0 + 32), acc + 32);
          tmem_ld_wait();
          uint8_t* rowp = sl + static_cast<uint32_t>(c0 / 64) * (BM * 128u) + row_off;
          if (last) {
            epilogue_row64<kActNone>(acc, rowp, row_sw);
          } else {
            epilogue_row64<kAct>(acc, rowp, row_sw);
          }
          // These accumulator columns have been read: seed them with the next bias.
          if (pre) {
            preload_bias32(tmem_row, bnext, c0);
            preload_bias32(tmem_row, bnext, c0 + 32);
          }
        }
      }
      if (pre) tmem_st_wait();
      if (npend > 0) {
        // The stores this warp issued a stage ago have read their slots; the
        // last of the four warps to release a slot refills it.
        if (lane == 0) {
          bulk_wait_group_read<0>();
#pragma unroll
          for (int a = 0; a < 2; ++a) {
            if (a >= npend) break;
            if (smem_atomic_add_acq_rel(free_cnt(pend_slot[a]), 1) % 4 == 3) {
              const int nt = pend_tile[a] + S;  // lands in the same slot
              if (nt < my_tiles) {
                mbar_arrive_expect_tx(x_full(pend_slot[a]), xbytes);
                for (int c = 0; c < p.D / 64; ++c)
                  tma_load_2d(base + slot_addr(pend_slot[a]) + static_cast<uint32_t>(c) * BM * 128u, &p.x_map,
                              x_full(pend_slot[a]), c * 64, tile_row(nt));
              }
              if (nt + kPrefetchAhead < my_tiles) prefetch_tile(nt + kPrefetchAhead);
            }
          }
        }
        npend = 0;
      }
      // TMEM reads (and bias writes) done, slot rows rewritten: publish.
      tc_fence_before_sync();
      fence_proxy_async_smem();
      __syncwarp();
      int ns[2], np[2];
#pragma unroll
      for (int a = 0; a < 2; ++a) {
        ns[a] = gs[a] + V;
        np[a] = gp[a];
        if (ns[a] >= S) {
          ns[a] -= S;
          np[a] ^= 1;
        }
      }
      if (lane == 0) {
        if (last) {
          // This warp's 32 rows of each finished tile go out by TMA.
#pragma unroll
          for (int a = 0; a < 2; ++a) {
            if (a >= na) break;
            const uint32_t slot_a = base + slot_addr(gs[a]);
            for (int c = 0; c < p.H / 64; ++c)
              tma_store_2d(&p.out_map, slot_a + static_cast<uint32_t>(c) * BM * 128u + 32u * q * 128u, c * 64,
                           tile_row(first + a) + static_cast<int>(32u * q));
          }
          bulk_commit_group();
        }
        // The last warp done with this stage issues the worker's next one.
        if (smem_atomic_add_acq_rel(ready_cnt(g), 1) % 4 == 3) {
          if (!last) {
            tc_fence_after_sync();
#pragma unroll
            for (int a = 0; a < 2; ++a) {
              if (a >= na) break;
              issue_mmas(g * P + a, gs[a], l + 1);
            }
            tc_commit(mma_done(g));
          } else if (first + V < my_tiles) {
            const int nna = my_tiles - first - V < P ? my_tiles - first - V : P;
            tc_fence_after_sync();
#pragma unroll
            for (int a = 0; a < 2; ++a) {
              if (a >= nna) break;
              ok = ok && mbar_wait(x_full(ns[a]), static_cast<uint32_t>(np[a]), p.err, kErrWaitMlp);
              if (ok) issue_mmas(g * P + a, ns[a], 0);
            }
            tc_commit(mma_done(g));
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (last) {
#pragma unroll
        for (int a = 0; a < 2; ++a) {
          pend_slot[a] = gs[a];
          pend_tile[a] = first + a;
          gs[a] = ns[a];
          gp[a] = np[a];
        }
        npend = na;
      }
    }
  }
  if (lane == 0) {
    bulk_wait_group<0>();
#pragma unroll
    for (int a = 0; a < 2; ++a)
      if (a < npend) smem_atomic_add_acq_rel(free_cnt(pend_slot[a]), 1);
  }
  __syncwarp();

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
  // Most row tiles in flight (V = workers x tiles per group) that fit TMEM
  // (V H columns) and shared memory with a ring of at least V + P slots (the
  // tiles in flight plus one group being loaded); fewer tiles per group first.
  int E = 0, P = 0, S = 0;
  for (int v = kMaxVirtual; v >= 1 && E == 0; --v) {
    if (v * H > 512) continue;
    for (int pp = 1; pp <= 2 && E == 0; ++pp) {
      if (v % pp != 0 || v / pp > kMaxWorkers) continue;
      for (int sl = kMaxSlots; sl >= v + pp; --sl) {
        if (make_layout(D, H, L, v, sl).alloc_bytes <= kSmemLimit) {
          E = v / pp;
          P = pp;
          S = sl;
          break;
        }
      }
    }
  }
  if (E == 0) return cudaErrorNotSupported;
  const Layout lo = make_layout(D, H, L, E * P, S);
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
  p.workers = E;
  p.pp = P;
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
