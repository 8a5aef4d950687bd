// Chained MLP in one persistent kernel on the tcgen05 tensor cores (sm_103a).
//
//   h_0 = x,  h_l = act(h_{l-1} . W_l + b_l) for l < L,  out = h_{L-1} . W_L + b_L
//
// x is [rows, D], W_1 [D, H], W_l [H, H], the last W [H, O] (or [D, O] when
// L = 1): O = H is the pages' form, O != H lets the chain end at another width.
// Operands are fp16 or bf16 with fp32 accumulation.
//
// The chained MLP of the "MLP Megakernel" README ("Architecture": 3- and
// 5-layer softplus MLPs; "Key ideas": all GEMMs and activations in one
// kernel, intermediates never reach global memory, a persistent kernel that
// walks row tiles round-robin, fp16 tensor-core operands with fp32
// accumulation and conversion to fp16 only at tile boundaries).
//
// Design (one CTA per SM, three kinds of warp):
//   * All L weight matrices stay resident in shared memory for the whole
//     launch (loaded once by TMA in the MN-major, 128-B-swizzled layout the
//     MMA reads); biases are kept as fp32.  Weights beyond kWeightBudget (or
//     leaving no room for the tile ring) are streamed instead: a loader warp
//     refills a ring of chunk slots of 64 rows of one layer's W each, and a
//     single MMA warp lets each chunk serve every accumulator of the round.
//   * Row tiles of 128 rows are loaded by TMA into a ring of S shared-memory
//     slots of 128 x max(D, H) fp16; CTA-local tile i uses slot i mod S.  V
//     row tiles are in flight.  Accumulator v owns TMEM columns
//     [v Hd, v Hd + Hd) for the fp32 layer result D_v (Hd = max(H, O)) and
//     [V Hd + v H/2, V Hd + v H/2 + H/2) for the 16-bit layer input (so every
//     region starts at a multiple of its own width), and the tiles v, v + V,
//     v + 2V, ...
//   * Layer 0 reads its A operand (x) from the slot; every later layer reads
//     it from TMEM, where the epilogue left the previous layer's activations
//     (row m in lane m, two 16-bit values per column).  Inter-layer
//     activations therefore never touch shared memory: the MMAs' shared-
//     memory traffic is the weights alone, which leaves the shared-memory
//     bandwidth that a 64- or 128-wide MMA otherwise saturates to the loads
//     and stores.
//   * MMA warps issue every tcgen05.mma; MMA warp j serves the accumulators
//     v = j mod (number of MMA warps).  An MMA issue blocks until the tensor
//     pipe takes it, and a burst of a layer's MMAs costs several hundred
//     cycles of issue latency, so no warp with epilogue work ever issues one
//     and several issuers let their bursts overlap in the pipe.  For each
//     (round, layer, own accumulator) in order an MMA warp waits until the
//     epilogue has released the accumulator (act_ready) and, for layer 0, the
//     tile has landed (x_full), then issues the layer's K / 16 MMAs
//     (M = 128, N = H) and commits them to mma_done.
//   * V epilogue workers of 4 C warps each own one accumulator; warp w of
//     a worker reads TMEM lane quarter w mod 4 (32 rows) and column group
//     (w / 4) mod C (H / C columns).  Per stage it waits for mma_done, reads
//     its accumulator columns (tcgen05.ld), rounds them to fp16, applies the
//     activation and writes them into the TMEM input region with tcgen05.st
//     (layers before the last), or, after the last layer, writes the output
//     rows into the tile's slot in the 128-B-swizzled layout and stores them
//     with TMA.  At its next stage, once that store has read the slot, it
//     releases its share of the slot (slot_free).
//   * One I/O warp refills each released slot with the tile due there next
//     and prefetches a later tile into L2, so HBM latency stays off the
//     critical path.
//   * The bias never costs an epilogue instruction per value: as soon as a
//     warp has read its accumulator columns it writes the NEXT layer's bias
//     (fp32) into them with tcgen05.st, and the next MMA accumulates on top.
//   * For training (coalesce_mlp_forward_train) every intermediate
//     activation h_l is also written to the caller's buffer: the epilogue
//     writes it into the tile's slot too (free after layer 0's MMA) and
//     TMA-stores its rows; before the slot is written again the store must
//     have read it.
//   * With fp16 operands softplus runs on packed fp16 pairs (one
//     ex2.approx.f16x2 plus a short polynomial); with bf16 operands, whose
//     8-bit significand would make that polynomial too coarse, every
//     activation is evaluated in fp32 and rounded to bf16.
// Ragged row tails are handled by TMA (zero-filled loads, clipped stores), and
// so are widths that are not multiples of 64: the kernel runs on widths
// rounded up to 64, the padded columns of x and W (and the padded rows of W)
// load as zeros, the padded bias entries are zero, so padded result columns
// hold 0 (act(0) after the activation) and meet only zero rows of the next W,
// and stores clip them.
// Every wait is bounded; a wait that runs out records an error and its warp
// stops, and the MMA warp drains its MMAs before TMEM is released.
#include <type_traits>

#include "epilogue.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace coalesce {
namespace mlp {

constexpr int BM = 128;
constexpr int kMaxLayers = 8;
constexpr int kMaxEpiWarps = 16;      // epilogue warps (4 C E)
constexpr int kMaxSlots = 12;
// Tiles prefetched into L2 beyond the ring.  Measured on the 3-layer 128-wide
// chain (means of 300 flushed calls): 0, 1, 2, 3, 4 and 8 tiles ahead gave
// 112.2, 112.2, 112.1, 112.6, 112.8 and 125.6 us; the 5-layer chain is flat.
constexpr int kPrefetchAhead = 2;
// With the activations stored, each tile writes (L-1) h tiles besides its
// output; that write stream evicted x tiles prefetched 4 ahead before they were
// loaded (1.5x the x bytes read from DRAM), so that form prefetches one ahead.
constexpr int kPrefetchAheadStoreH = 1;
constexpr uint32_t kSmemLimit = 232448 - 64;  // opt-in maximum per block, less the static shared memory
constexpr uint32_t kWeightBudget = 160u * 1024u;  // resident weights; beyond it they are streamed
constexpr uint32_t kChunkBlock = 64u * 128u;        // one 64-row x 64-column block of a streamed chunk
constexpr int kMaxWeightSlots = 4;

// Shared-memory plan, identical on host and device.  Small items (barriers,
// TMEM address, fp32 biases) sit at the start of the dynamic window; the
// swizzled operand buffers start at the next 1 KiB boundary after them.
struct Layout {
  // relative to the start of dynamic shared memory
  uint32_t bar_off;        // w_full, drain, x_full[S], slot_free[S], mma_done[V], act_ready[V], wc_full[WR], wc_free[WR]
  uint32_t tmem_slot_off;
  uint32_t bias_off;
  uint32_t small_bytes;
  // relative to the 1 KiB-aligned big base
  uint32_t w_off[kMaxLayers];  // resident weights
  uint32_t wring_off;      // streamed weights: WR chunk slots of 64 rows of one layer's W
  uint32_t wchunk_bytes;
  uint32_t wslots;         // WR (0: weights resident)
  uint32_t slot_off;       // slot s at slot_off + s * slot_bytes
  uint32_t slots;          // S
  uint32_t slot_bytes;
  uint32_t big_bytes;
  uint32_t alloc_bytes;    // small + worst-case alignment padding + big
  uint32_t in_col0;        // first TMEM column of the fp16 input regions (V H)
  uint32_t tmem_cols;      // allocated TMEM columns (power of two)
};

__host__ __device__ inline uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// Output width of layer l (0-based) of an L-layer chain.
__host__ __device__ inline int layer_out(int H, int O, int L, int l) { return l == L - 1 ? O : H; }

// V row tiles in flight (V accumulators), S slots; WR > 0 streams the
// weights through WR chunk slots instead of keeping them resident.
__host__ __device__ inline Layout make_layout(int D, int H, int O, int L, int V, int S, int WR = 0) {
  Layout lo{};
  uint32_t off = 0;
  lo.bar_off = off;
  off += 8u * (2u + 2u * static_cast<uint32_t>(S + V + WR));
  lo.tmem_slot_off = off;
  off += 16;
  const int Hd = H > O ? H : O;
  lo.bias_off = align_up(off, 16);  // read as float4; layer l's bias at l * Hd
  off = lo.bias_off + static_cast<uint32_t>(L * Hd) * 4u;
  lo.small_bytes = align_up(off, 16);
  uint32_t big = 0;
  lo.wslots = static_cast<uint32_t>(WR);
  if (WR == 0) {
    for (int l = 0; l < L; ++l) {
      const uint32_t K = l == 0 ? D : H;
      lo.w_off[l] = big;
      big += static_cast<uint32_t>(layer_out(H, O, L, l) / 64) * K * 128u;
    }
  } else {
    lo.wring_off = 0;
    lo.wchunk_bytes = static_cast<uint32_t>(Hd / 64) * kChunkBlock;
    big = static_cast<uint32_t>(WR) * lo.wchunk_bytes;
  }
  const int kmax = D > Hd ? D : Hd;
  lo.slot_bytes = static_cast<uint32_t>(kmax / 64) * BM * 128u;
  lo.slot_off = big;
  lo.slots = static_cast<uint32_t>(S);
  big += static_cast<uint32_t>(S) * lo.slot_bytes;
  lo.big_bytes = big;
  // dynamic shared memory is at least 16-byte aligned: at most 1008 bytes of padding
  lo.alloc_bytes = lo.small_bytes + 1008u + big;
  lo.in_col0 = static_cast<uint32_t>(V * Hd);
  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>(V * Hd + V * H / 2)) cols <<= 1;
  lo.tmem_cols = cols;
  return lo;
}

struct Params {
  CUtensorMap x_map;                  // x [rows, D], box 128 x 64, 128-B swizzle
  CUtensorMap out_map;                // out [rows, O], box 32 x 64, 128-B swizzle
  CUtensorMap w_map[kMaxLayers];      // W_l [K_l, N_l], box K_l x 64 (64 x 64 when streamed), 128-B swizzle
  CUtensorMap h_map[kMaxLayers - 1];  // h_l [rows, H] (store_h only), box 32 x 64, 128-B swizzle
  const uint16_t* bias[kMaxLayers];   // b_l[N_l] (fp16 or bf16 bits), or nullptr
  int nb[kMaxLayers];                 // entries of b_l: the caller's N_l (D, H and O below are padded)
  Layout lo;                          // shared-memory plan (host-computed)
  int rows, D, H, O, L;                // widths rounded up to multiples of 64
  int workers;                        // V: epilogue workers, one accumulator (row tile in flight) each
  int cgroups;                        // C: column groups per accumulator (warps per worker = 4 C)
  int cshift;                         // log2(C): C is 1, 2 or 4
  int mma_warps;                      // warps that issue MMAs (<= V); one I/O warp follows them
  int store_h;                        // also store every intermediate activation (h_map)
  uint32_t* err;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// fp32 accumulator columns -> 16-bit pairs with the activation applied.
template <int kAct, bool kBf16>
__device__ __forceinline__ uint32_t act_pair(uint32_t lo_bits, uint32_t hi_bits) {
  const float lo = __uint_as_float(lo_bits);
  const float hi = __uint_as_float(hi_bits);
  if constexpr (kBf16) {
    return pack_bf16x2(act_apply_16<kAct>(lo), act_apply_16<kAct>(hi));
  } else if constexpr (kAct == kActSoftplus) {
    return softplus_f16x2(pack_f16x2(lo, hi));
  } else if constexpr (kAct == kActNone) {
    return pack_f16x2(lo, hi);
  } else {
    return pack_f16x2(act_apply<kAct>(lo), act_apply<kAct>(hi));
  }
}

// Write bias[c0 .. c0+31] (fp32, shared memory) into this warp's 32 TMEM lanes
// at `taddr` (32 columns), so that the next MMA adds onto it.
__device__ __forceinline__ void preload_bias32(uint32_t taddr, const float* bias_c0) {
  uint32_t b[32];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 v = *reinterpret_cast<const float4*>(bias_c0 + 4 * i);
    b[4 * i] = __float_as_uint(v.x);
    b[4 * i + 1] = __float_as_uint(v.y);
    b[4 * i + 2] = __float_as_uint(v.z);
    b[4 * i + 3] = __float_as_uint(v.w);
  }
  tmem_st_32x32b_x32(taddr, b);
}

// One layer's MMAs for one row tile, KS k-steps of 16.  The weights W are the
// B operand (MN-major, 64-column blocks of K rows x 128 B).  For layer 0 the
// A operand is the tile's slot (K-major, 64-column blocks of 128 rows x
// 128 B; `a` is its smem descriptor); later layers take A from TMEM (`a` is
// the TMEM address of the fp16 input region; k-step ks is 8 columns on).
// The smem descriptors of later k-steps differ from the first only in the
// start-address field (bits 0..13, address >> 4), so they are formed by
// adding the byte offset >> 4 to the first.
template <int KS, bool kFromTmem>
__device__ __forceinline__ void issue_layer(uint32_t d, uint64_t a, uint64_t b_desc, uint32_t idesc, uint32_t acc0) {
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    const uint64_t bd = b_desc + static_cast<uint64_t>((ks * 2048) >> 4);
    const uint32_t acc = ks > 0 ? 1u : acc0;
    if constexpr (kFromTmem) {
      tc_mma_f16_ts(d, static_cast<uint32_t>(a) + 8u * ks, bd, idesc, acc);
    } else {
      const uint64_t ad = a + static_cast<uint64_t>(((ks / 4) * BM * 128 + (ks % 4) * 32) >> 4);
      tc_mma_f16(d, ad, bd, idesc, acc);
    }
  }
}

template <bool kFromTmem>
__device__ __forceinline__ void issue_layer_k(int K, uint32_t d, uint64_t a, uint64_t b_desc, uint32_t idesc,
                                              uint32_t acc0) {
  switch (K / 16) {
    case 4: issue_layer<4, kFromTmem>(d, a, b_desc, idesc, acc0); break;
    case 8: issue_layer<8, kFromTmem>(d, a, b_desc, idesc, acc0); break;
    case 12: issue_layer<12, kFromTmem>(d, a, b_desc, idesc, acc0); break;
    default: issue_layer<16, kFromTmem>(d, a, b_desc, idesc, acc0); break;
  }
}

// 20 warps at most (16 epilogue, up to 3 MMA, 1 I/O): an SM sub-partition
// holds five of them, which must fit 5 x 32 x 96 registers in its 16 K-entry
// register file.
// kSquare: O = H (every layer H wide), known at compile time so that the
// per-layer column ranges fold away.
// kStoreH: also store every intermediate activation (training forward).
// kLog2: an fp16 softplus chain that carries its activations in log2 units
// (softplus_log2_f16x2): log2 e is applied to layer 0's result, ln 2 to the
// last layer's, and the biases of layers 1 .. L-1 are held times log2 e.
// kFold (resident weights only): the two factors are folded into W_0 and
// W_{L-1} in shared memory instead, once per CTA, so that the first and last
// layers' results need no multiply; then the biases of layers 0 .. L-2 are
// held times log2 e.
__device__ __forceinline__ void named_barrier_arrive(uint32_t id, uint32_t count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

template <int kAct, bool kBf16, bool kSquare, bool kStoreH, bool kLog2 = false, bool kFold = false>
__global__ void __maxnreg__(96) mlp_fused_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ int bias_nonzero[kMaxLayers];
  const int E = p.workers;
  const int C = p.cgroups;
  const int V = E;  // one accumulator (row tile in flight) per worker
  const Layout& lo = p.lo;
  const int S = static_cast<int>(lo.slots);
  const uint32_t sbase = smem_u32(smem_raw);                        // small items
  const uint32_t base = (sbase + lo.small_bytes + 1023u) & ~1023u;  // swizzled buffers
  uint8_t* gbase = smem_raw + (base - sbase);
  const uint32_t warp = warp_index_uniform();
  const uint32_t lane = threadIdx.x % 32;
  const uint32_t epi_warps = 4u * static_cast<uint32_t>(C * E);
  const uint32_t worker_warps = 4u * static_cast<uint32_t>(C);
  const int O = kSquare ? p.H : p.O;
  const int Hd = p.H > O ? p.H : O;  // TMEM columns of each layer result
  const int num_tiles = (p.rows + BM - 1) / BM;
  // tiles of this CTA: blockIdx.x + i * gridDim.x, i = 0 .. my_tiles - 1
  const int my_tiles = blockIdx.x < num_tiles ? (num_tiles - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;

  const uint32_t w_full = sbase + lo.bar_off;
  const uint32_t drain = w_full + 8u;
  auto x_full = [&](int s) { return sbase + lo.bar_off + 8u * (2 + s); };
  auto slot_free = [&](int s) { return sbase + lo.bar_off + 8u * (2 + S + s); };
  auto mma_done = [&](int v) { return sbase + lo.bar_off + 8u * (2 + 2 * S + v); };
  auto act_ready = [&](int v) { return sbase + lo.bar_off + 8u * (2 + 2 * S + V + v); };
  const int WR = static_cast<int>(lo.wslots);
  auto wc_full = [&](int i) { return sbase + lo.bar_off + 8u * (2 + 2 * S + 2 * V + i); };
  auto wc_free = [&](int i) { return sbase + lo.bar_off + 8u * (2 + 2 * S + 2 * V + WR + i); };
  const uint32_t io_warp = epi_warps + static_cast<uint32_t>(p.mma_warps);
  auto slot_addr = [&](int s) { return lo.slot_off + static_cast<uint32_t>(s) * lo.slot_bytes; };
  auto tile_row = [&](int i) { return (static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x)) * BM; };
  const uint32_t xbytes = static_cast<uint32_t>(p.D) * BM * 2u;
  constexpr int kAhead = kStoreH ? kPrefetchAheadStoreH : kPrefetchAhead;
  auto prefetch_tile = [&](int i) {
    for (int c = 0; c < p.D / 64; ++c) tma_prefetch_l2_2d(&p.x_map, c * 64, tile_row(i));
  };
  auto load_tile = [&](int i, int s) {
    mbar_arrive_expect_tx(x_full(s), xbytes);
    for (int c = 0; c < p.D / 64; ++c)
      tma_load_2d(base + slot_addr(s) + static_cast<uint32_t>(c) * BM * 128u, &p.x_map, x_full(s), c * 64,
                  tile_row(i));
  };

  // ---- set-up: barriers, TMEM, biases (fp32), weights and the first S tiles (TMA)
  if (threadIdx.x == 0) {
    mbar_init(w_full, 1);
    mbar_init(drain, static_cast<uint32_t>(p.mma_warps));
    for (int s = 0; s < S; ++s) {
      mbar_init(x_full(s), 1);
      mbar_init(slot_free(s), worker_warps);  // every warp of the tile's worker
    }
    for (int v = 0; v < V; ++v) {
      mbar_init(mma_done(v), 1);
      mbar_init(act_ready(v), worker_warps);
    }
    for (int i = 0; i < WR; ++i) {
      mbar_init(wc_full(i), 1);
      mbar_init(wc_free(i), 1);
    }
    fence_mbarrier_init();
  }
  if (warp == 0) {
    tmem_alloc(sbase + lo.tmem_slot_off, lo.tmem_cols);
    tmem_relinquish_alloc_permit();
  }
  float* bias_s = reinterpret_cast<float*>(smem_raw + lo.bias_off);
  if (threadIdx.x < kMaxLayers) bias_nonzero[threadIdx.x] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < p.L * Hd; i += blockDim.x) {
    const int l = i / Hd, n = i % Hd;
    float v = 0.0f;
    if (p.bias[l] != nullptr && n < p.nb[l]) {
      const uint16_t bits = p.bias[l][n];
      v = kBf16 ? __bfloat162float(__ushort_as_bfloat16(bits)) : __half2float(__ushort_as_half(bits));
    }
    // log2 units: every layer's bias but the last times log2 e when the first
    // layer's weights carry the factor (kFold), else every bias but the first
    if (kLog2 && (kFold ? l < p.L - 1 : l > 0)) v *= kLog2e;
    bias_s[i] = v;
    if (v != 0.0f) bias_nonzero[l] = 1;  // benign race: every writer stores 1
  }
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&p.x_map);
    tma_prefetch_desc(&p.out_map);
    if (WR == 0) {
      uint32_t wbytes = 0;
      for (int l = 0; l < p.L; ++l)
        wbytes += static_cast<uint32_t>(layer_out(p.H, O, p.L, l) / 64) * (l == 0 ? p.D : p.H) * 128u;
      mbar_arrive_expect_tx(w_full, wbytes);
      for (int l = 0; l < p.L; ++l) {
        const int K = l == 0 ? p.D : p.H;
        for (int j = 0; j < layer_out(p.H, O, p.L, l) / 64; ++j)
          tma_load_2d(base + lo.w_off[l] + static_cast<uint32_t>(j * K) * 128u, &p.w_map[l], w_full, j * 64, 0);
      }
    }
    for (int i = 0; i < S && i < my_tiles; ++i) load_tile(i, i);  // tile i -> slot i
    for (int i = S; i < S + kAhead && i < my_tiles; ++i) prefetch_tile(i);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem_raw + lo.tmem_slot_off);

  if (warp == io_warp) {
    // ---------------------------------------------------------------- slot refills
    if (lane == 0) {
      int s = 0;
      uint32_t fp = 0;
      for (int i = 0; i + S < my_tiles; ++i) {
        if (!mbar_wait(slot_free(s), fp, p.err, kErrWaitMlp)) break;
        load_tile(i + S, s);
        if (i + S + kAhead < my_tiles) prefetch_tile(i + S + kAhead);
        if (++s == S) {
          s = 0;
          fp ^= 1u;
        }
      }
    }
    __syncwarp();
  } else if (WR > 0 && warp == io_warp + 1) {
    // ---------------------------------------------------------------- streamed weights
    // Every round (V tiles) takes each layer's W in 64-row chunks, in the
    // order the MMA warp consumes them; a chunk slot is refilled once the
    // MMAs that read it have completed.
    if (lane == 0) {
      int ws = 0;
      uint32_t wph = 0;
      bool wrapped = false, ok = true;
      for (int m = 0; ok && m * V < my_tiles; ++m) {
        for (int l = 0; ok && l < p.L; ++l) {
          const int K = l == 0 ? p.D : p.H;
          const int N = layer_out(p.H, O, p.L, l);
          for (int c = 0; c < K / 64; ++c) {
            if (wrapped && !mbar_wait(wc_free(ws), wph ^ 1u, p.err, kErrWaitMlp)) {
              ok = false;
              break;
            }
            const uint32_t dst = base + lo.wring_off + static_cast<uint32_t>(ws) * lo.wchunk_bytes;
            mbar_arrive_expect_tx(wc_full(ws), static_cast<uint32_t>(N / 64) * kChunkBlock);
            for (int jb = 0; jb < N / 64; ++jb)
              tma_load_2d(dst + static_cast<uint32_t>(jb) * kChunkBlock, &p.w_map[l], wc_full(ws), jb * 64, c * 64);
            if (++ws == WR) {
              ws = 0;
              wph ^= 1u;
              wrapped = true;
            }
          }
        }
      }
    }
    __syncwarp();
  } else if (WR > 0 && warp >= epi_warps) {
    // ---------------------------------------------------------------- MMA issuer, streamed weights
    // One MMA warp.  Per round and layer every accumulator must be ready;
    // then each 64-row chunk of W_l (four k-steps) serves all of them in turn
    // and is released by a commit, and the last chunk's commit publishes the
    // accumulators.
    bool ok = true;
    uint32_t apar = 0;
    int s0 = 0;
    uint32_t x0 = 0;
    int ws = 0;
    uint32_t wph = 0;
    for (int m = 0; ok && m * V < my_tiles; ++m) {
      const int nv = my_tiles - m * V < V ? my_tiles - m * V : V;
      for (int l = 0; ok && l < p.L; ++l) {
        const int K = l == 0 ? p.D : p.H;
        const uint32_t idesc =
            idesc_f16_f32acc(kBf16, false, true, BM, static_cast<uint32_t>(layer_out(p.H, O, p.L, l)));
        const uint32_t acc0 = bias_nonzero[l] ? 1u : 0u;
        for (int v = 0; ok && v < nv; ++v) {
          const int s = s0 + v < S ? s0 + v : s0 + v - S;
          const uint32_t xp = s0 + v < S ? x0 : x0 ^ 1u;
          ok = mbar_wait(act_ready(v), (apar >> v) & 1u, p.err, kErrWaitMlp);
          apar ^= 1u << v;
          if (ok && l == 0) ok = mbar_wait(x_full(s), xp, p.err, kErrWaitMlp);
        }
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        for (int c = 0; ok && c < K / 64; ++c) {
          ok = mbar_wait(wc_full(ws), wph, p.err, kErrWaitMlp);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          if (elect_one()) {
            // chunk: 64-column blocks of 64 k-rows x 128 B, kChunkBlock apart (MN-major B)
            const uint64_t bd0 = smem_desc_sw128(base + lo.wring_off + static_cast<uint32_t>(ws) * lo.wchunk_bytes,
                                                 kChunkBlock, 1024);
            for (int v = 0; v < nv; ++v) {
              const uint32_t d = tmem_base + static_cast<uint32_t>(v * Hd);
              const int s = s0 + v < S ? s0 + v : s0 + v - S;
#pragma unroll
              for (int k4 = 0; k4 < 4; ++k4) {
                const int ks = 4 * c + k4;
                const uint64_t bd = bd0 + static_cast<uint64_t>((k4 * 2048) >> 4);
                const uint32_t acc = ks > 0 ? 1u : acc0;
                if (l == 0) {
                  const uint64_t ad = smem_desc_sw128(base + slot_addr(s), 16, 1024) +
                                      static_cast<uint64_t>((c * BM * 128 + k4 * 32) >> 4);
                  tc_mma_f16(d, ad, bd, idesc, acc);
                } else {
                  const uint32_t a_in = tmem_base + lo.in_col0 + static_cast<uint32_t>(v * (p.H / 2));
                  tc_mma_f16_ts(d, a_in + 8u * static_cast<uint32_t>(ks), bd, idesc, acc);
                }
              }
            }
            tc_commit(wc_free(ws));
            if (c == K / 64 - 1)
              for (int v = 0; v < nv; ++v) tc_commit(mma_done(v));
          }
          __syncwarp();
          if (++ws == WR) {
            ws = 0;
            wph ^= 1u;
          }
        }
      }
      s0 += V;
      if (s0 >= S) {
        s0 -= S;
        x0 ^= 1u;
      }
    }
    if (elect_one()) tc_commit(drain);
    __syncwarp();
    mbar_wait(drain, 0, p.err, kErrWaitMlp);
  } else if (warp >= epi_warps) {
    // ---------------------------------------------------------------- MMA issuers
    // The whole warp walks the schedule (so descriptors are warp-uniform);
    // one elected lane issues.
    const int j = static_cast<int>(warp - epi_warps);
    const int nm = p.mma_warps;
    bool ok = mbar_wait(w_full, 0, p.err, kErrWaitMlp);
    // the epilogue warps fold the unit factors into W_0 and W_{L-1} first (kFold)
    if constexpr (kLog2 && kFold) named_barrier_sync(2, (epi_warps + static_cast<uint32_t>(p.mma_warps)) * 32u);
    uint32_t apar = 0;  // bit v: parity of the next act_ready[v] phase
    int s0 = 0;         // slot of tile m V (the round's first tile)
    uint32_t x0 = 0;    // load parity of that slot's current tile
    for (int m = 0; ok && m * V < my_tiles; ++m) {
      for (int l = 0; ok && l < p.L; ++l) {
        const int K = l == 0 ? p.D : p.H;
        const uint32_t idesc =
            idesc_f16_f32acc(kBf16, false, true, BM, static_cast<uint32_t>(layer_out(p.H, O, p.L, l)));
        const uint64_t b_desc = smem_desc_sw128(base + lo.w_off[l], static_cast<uint32_t>(K) * 128u, 1024);
        const uint32_t acc0 = bias_nonzero[l] ? 1u : 0u;
        for (int v = j; v < V; v += nm) {
          if (m * V + v >= my_tiles) break;
          // tile m V + v sits in slot s0 + v (V < S: one wrap at most)
          const int s = s0 + v < S ? s0 + v : s0 + v - S;
          const uint32_t xp = s0 + v < S ? x0 : x0 ^ 1u;
          ok = mbar_wait(act_ready(v), (apar >> v) & 1u, p.err, kErrWaitMlp);
          apar ^= 1u << v;
          if (ok && l == 0) ok = mbar_wait(x_full(s), xp, p.err, kErrWaitMlp);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t d = tmem_base + static_cast<uint32_t>(v * Hd);
          if (elect_one()) {
            if (l == 0) {
              issue_layer_k<false>(K, d, smem_desc_sw128(base + slot_addr(s), 16, 1024), b_desc, idesc, acc0);
            } else {
              const uint32_t a_in = tmem_base + lo.in_col0 + static_cast<uint32_t>(v * (p.H / 2));
              issue_layer_k<true>(K, d, a_in, b_desc, idesc, acc0);
            }
            tc_commit(mma_done(v));
          }
          __syncwarp();
        }
      }
      // next round: its first tile is V slots further on (V < S: one wrap at most)
      s0 += V;
      if (s0 >= S) {
        s0 -= S;
        x0 ^= 1u;
      }
    }
    // Every MMA issued above has completed before TMEM can be released.
    if (elect_one()) tc_commit(drain);
    __syncwarp();
    mbar_wait(drain, 0, p.err, kErrWaitMlp);
  } else {
    // ---------------------------------------------------------------- epilogue workers
    // Worker g (4 C warps) owns accumulator g and the CTA-local tiles g,
    // g + V, g + 2V, ...  The stage loop is kept lean: barrier and TMEM
    // addresses are formed once, single-lane actions (barrier arrivals, TMA
    // stores, bulk-group waits) are predicated on `leader` instead of
    // branched, a wait costs one try_wait when its phase has completed, and
    // every layer width is a multiple of 64, so columns go in 64-column
    // pieces of two unrolled 32-column TMEM round trips.
    const int g = static_cast<int>(warp / worker_warps);
    const uint32_t q = warp & 3u;                                   // TMEM lane quarter of this warp
    const int cg = static_cast<int>((warp >> 2) & static_cast<uint32_t>(C - 1));  // column group of this warp
    const uint32_t leader = lane == 0 ? 1u : 0u;
    const uint32_t row = 32u * q + lane;                            // row within the tile (= TMEM lane)
    const uint32_t row_sw = row & 7u;
    const uint32_t lane_base = (32u * q) << 16;
    const uint32_t dcol = tmem_base + lane_base + static_cast<uint32_t>(g * Hd);  // D_g, column 0
    const uint32_t acol = tmem_base + lane_base + lo.in_col0 + static_cast<uint32_t>(g * (p.H / 2));
    const uint32_t done_bar = mma_done(g);
    const uint32_t ready_bar = act_ready(g);
    if constexpr (kLog2 && kFold) {
      // Fold the chain's unit changes into the resident weights, once: W_0
      // times log2 e (its result then comes out in log2 units) and W_{L-1}
      // times ln 2 (its result in natural units), each weight times the fp32
      // factor and rounded once to fp16.  The epilogue warps share the work,
      // make it visible to the tensor cores and release the MMA warps.
      bool okw = mbar_wait_warp(w_full, 0, p.err, kErrWaitMlp);
      if (okw) {
        auto scale = [](__half2 w, float f) {
          const float2 v = __half22float2(w);
          return __floats2half2_rn(v.x * f, v.y * f);
        };
        const int nthr = static_cast<int>(epi_warps) * 32;
        const int me = static_cast<int>(warp) * 32 + static_cast<int>(lane);
        __half2* w0 = reinterpret_cast<__half2*>(gbase + lo.w_off[0]);
        __half2* w1 = reinterpret_cast<__half2*>(gbase + lo.w_off[p.L - 1]);
        const int nw0 = layer_out(p.H, O, p.L, 0) * p.D / 2;
        const int nw1 = layer_out(p.H, O, p.L, p.L - 1) * p.H / 2;
        for (int i = me; i < nw0; i += nthr) w0[i] = scale(w0[i], kLog2e);
        for (int i = me; i < nw1; i += nthr) w1[i] = scale(w1[i], kLn2);
        fence_proxy_async_smem();
      }
      named_barrier_arrive(2, (epi_warps + static_cast<uint32_t>(p.mma_warps)) * 32u);
    }
    uint32_t pre_mask = 0;  // bit l: layer l has a non-zero bias, seeded into TMEM before its MMA
    for (int l = 0; l < p.L; ++l) pre_mask |= bias_nonzero[l] ? 1u << l : 0u;
    // Every accumulator starts out holding b_0 for its first MMA.  A warp
    // seeds its column group of each layer's result (with C > 1 every layer
    // has the same width, so that is the range it reads).
    const int n0 = layer_out(p.H, O, p.L, 0) >> p.cshift;
    if (pre_mask & 1u) {
      for (int c0 = cg * n0; c0 < (cg + 1) * n0; c0 += 32) preload_bias32(dcol + static_cast<uint32_t>(c0), bias_s + c0);
      tmem_st_wait();
    }
    tc_fence_before_sync();
    __syncwarp();
    mbar_arrive_if(ready_bar, leader);
    uint32_t mpar = 0;   // parity of the next mma_done phase
    int pend_slot = -1;  // slot this warp last stored from, released at its next stage
    int s = g;           // slot of this worker's current tile (g < V < S)
    for (int t = g; t < my_tiles; t += V) {
      uint8_t* const slot_rows = gbase + slot_addr(s) + row * 128u;  // this thread's row of the slot, block 0
      const uint32_t slot_src = base + slot_addr(s) + 32u * q * 128u;  // this warp's 32 rows, block 0
      const int r0 = tile_row(t) + static_cast<int>(32u * q);
      // One layer of this tile; kLast (a compile-time tag) marks the chain's
      // last layer, whose result is the output.  False if a wait ran out.
      // kFirst marks layer 0 of a log2-unit chain whose factors are not folded
      // into the weights (see kLog2, kFold).
      auto stage = [&](auto first_tag, auto last_tag, int l) -> bool {
        constexpr bool first = decltype(first_tag)::value;
        constexpr bool last = decltype(last_tag)::value;
        const int next_l = last ? 0 : l + 1;  // the next MMA on this accumulator
        const bool pre = (pre_mask >> next_l) & 1u;
        const float* bnext = bias_s + next_l * Hd;
        const int cw = kSquare ? (p.H >> p.cshift) : (last ? O : p.H) >> p.cshift;  // columns per warp
        const int c_lo = cg * cw;
        const int nw = kSquare ? cw : layer_out(p.H, O, p.L, next_l) >> p.cshift;  // next layer's columns per warp
        const int n_lo = cg * nw;
        if (!mbar_wait_warp(done_bar, mpar, p.err, kErrWaitMlp)) return false;
        mpar ^= 1u;
        tc_fence_after_sync();
        if (kStoreH && l > 0) {
          // the slot still holds this tile's previous activation: its store must have read it
          if (leader) bulk_wait_group_read<0>();
          __syncwarp();
        }
#pragma unroll 1
        for (int c64 = c_lo; c64 < c_lo + cw; c64 += 64) {
          uint8_t* const rowp = slot_rows + static_cast<uint32_t>(c64 / 64) * (BM * 128u);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int c0 = c64 + 32 * j;
            uint32_t acc[32];
            tmem_ld_32x32b_x32(dcol + static_cast<uint32_t>(c0), acc);
            tmem_ld_wait();
            if constexpr (!last) {
              // next layer's A operand: row `row`, columns c0 .. c0+31 as 16 packed pairs
              uint32_t h[16];
#pragma unroll
              for (int k = 0; k < 16; ++k) {
                if constexpr (kLog2 && first && !kFold)
                  h[k] = softplus_log2_f16x2(scale_pack_f16x2(acc[2 * k], acc[2 * k + 1], kLog2e));
                else if constexpr (kLog2)
                  h[k] = softplus_log2_f16x2(act_pair<kActNone, false>(acc[2 * k], acc[2 * k + 1]));
                else
                  h[k] = act_pair<kAct, kBf16>(acc[2 * k], acc[2 * k + 1]);
              }
              tmem_st_32x32b_x16(acol + static_cast<uint32_t>(c0 / 2), h);
              if constexpr (kStoreH) {
                // the same values as rows of the slot, for the activation store
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  *reinterpret_cast<uint4*>(rowp + ((static_cast<uint32_t>(4 * j + i) ^ row_sw) << 4)) =
                      make_uint4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
              }
            } else {
              // output rows into the slot (128-B swizzle: 16-byte chunk i at i ^ (row & 7))
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                uint32_t w[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                  if constexpr (kLog2 && !first && !kFold)
                    w[k] = scale_pack_f16x2(acc[8 * i + 2 * k], acc[8 * i + 2 * k + 1], kLn2);
                  else
                    w[k] = act_pair<kActNone, kBf16>(acc[8 * i + 2 * k], acc[8 * i + 2 * k + 1]);
                }
                *reinterpret_cast<uint4*>(rowp + ((static_cast<uint32_t>(4 * j + i) ^ row_sw) << 4)) =
                    make_uint4(w[0], w[1], w[2], w[3]);
              }
            }
            // These accumulator columns have been read: seed them with the next bias.
            if (kSquare) {
              if (pre) preload_bias32(dcol + static_cast<uint32_t>(c0), bnext + c0);
            } else if (pre && c0 >= n_lo && c0 < n_lo + nw) {
              preload_bias32(dcol + static_cast<uint32_t>(c0), bnext + c0);
            }
          }
        }
        // A next layer wider than this one (C = 1 then): seed the columns
        // beyond this layer's width too; no MMA or warp uses them meanwhile.
        if (!kSquare && pre)
          for (int c0 = c_lo + cw > n_lo ? c_lo + cw : n_lo; c0 < n_lo + nw; c0 += 32)
            preload_bias32(dcol + static_cast<uint32_t>(c0), bnext + c0);
        tmem_st_wait();
        // The store this warp issued a stage ago has read its slot: release it.
        if (pend_slot >= 0) {
          bulk_read_done_arrive_if(slot_free(pend_slot), leader);
          pend_slot = -1;
        }
        // TMEM reads and writes done (and output rows written): publish.
        tc_fence_before_sync();
        if constexpr (last || kStoreH) fence_proxy_async_smem();
        __syncwarp();
        if constexpr (last || kStoreH) {
          // This warp's 32 rows x cw columns go out by TMA: h_{l+1}, or the finished tile.
          const CUtensorMap* map = last ? &p.out_map : &p.h_map[l];
          for (int c = c_lo; c < c_lo + cw; c += 64)
            tma_store_2d_if(map, slot_src + static_cast<uint32_t>(c / 64) * BM * 128u, c, r0, leader);
          bulk_commit_group_if(leader);
        }
        mbar_arrive_if(ready_bar, leader);
        if constexpr (last) pend_slot = s;
        return true;
      };
      if (p.L == 1) {
        if (!stage(std::bool_constant<kLog2>{}, std::true_type{}, 0)) goto epilogue_done;
      } else {
        if (!stage(std::bool_constant<kLog2 && !kFold>{}, std::false_type{}, 0)) goto epilogue_done;
        for (int l = 1; l < p.L - 1; ++l)
          if (!stage(std::false_type{}, std::false_type{}, l)) goto epilogue_done;
        if (!stage(std::false_type{}, std::true_type{}, p.L - 1)) goto epilogue_done;
      }
      s += V;
      if (s >= S) s -= S;
    }
  epilogue_done:
    if (leader) bulk_wait_group<0>();
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, lo.tmem_cols);
  }
}

}  // namespace mlp

cudaError_t launch_mlp_fused(const DeviceCtx& dev, int64_t rows, int Dt, int Ht, int Ot, int L, bool bf16,
                             const void* x, const void* const* W, const void* const* b, void* out, int act,
                             cudaStream_t stream, void* const* h) {
  using namespace mlp;
  // The caller's widths Dt, Ht, Ot (multiples of 8: 16-byte rows) are what the
  // tensor maps and bias reads use; the kernel's layout uses them rounded up
  // to multiples of 64.
  if (L > kMaxLayers || Dt % 8 != 0 || Ht % 8 != 0 || Ot % 8 != 0 || Dt < 1 || Ht < 1 || Ot < 1 || Dt > 256 ||
      Ht > 256 || Ot > 256)
    return cudaErrorNotSupported;
  const int D = (Dt + 63) / 64 * 64, H = (Ht + 63) / 64 * 64, O = (Ot + 63) / 64 * 64;
  const int Hd = H > O ? H : O;
  // Most row tiles in flight (V accumulators, one per worker, V <= 4) whose
  // TMEM regions (Hd + H/2 columns each) fit the 512 TMEM columns, with a ring
  // of at least V + 1 slots (the tiles in flight plus one being loaded) in
  // shared memory.  (Every width is at least 64, so at most five regions of
  // 96 or more columns fit; four is the most a multiple of the worker count
  // allows.)  Each worker has 4 C warps (C column groups of a multiple of 64
  // columns, C = 1 when O != H), as many as 16 epilogue warps allow.
  // Weights beyond kWeightBudget are streamed in 64-row chunks through at
  // least two chunk slots, by one loader warp, for one MMA warp serving at
  // most two accumulators.
  // They are streamed too when resident weights leave no room for the ring.
  uint64_t wtotal = 0;
  for (int l = 0; l < L; ++l) wtotal += 2ull * static_cast<uint64_t>(l == 0 ? D : H) * layer_out(H, O, L, l);
  int E = 0, S = 0, WR = 0;
  auto choose = [&](bool streamed) {
    for (int v = 4; v >= 1 && E == 0; --v) {
      if (v * (Hd + H / 2) > 512 || (streamed && v > 2)) continue;
      for (int sl = kMaxSlots; sl >= v + 1 && E == 0; --sl) {
        for (int wr = streamed ? kMaxWeightSlots : 0; wr >= (streamed ? 2 : 0); --wr) {
          if (make_layout(D, H, O, L, v, sl, wr).alloc_bytes <= kSmemLimit) {
            E = v;
            S = sl;
            WR = wr;
            break;
          }
        }
      }
    }
  };
  if (wtotal <= kWeightBudget) choose(false);
  if (E == 0) choose(true);
  if (E == 0) return cudaErrorNotSupported;
  const bool streamed = WR > 0;
  int C = 1;
  while (O == H && 4 * (2 * C) * E <= kMaxEpiWarps && (H / (2 * C)) % 64 == 0) C *= 2;
  // One MMA warp per two accumulators: a single issuer serialises the
  // bursts' issue latency, one per accumulator lets them collide.
  const int nm = E / 2 > 0 && !streamed ? E / 2 : 1;
  const Layout lo = make_layout(D, H, O, L, E, S, WR);
  const uint32_t smem = lo.alloc_bytes;
  if (lo.bias_off % 16 != 0 || lo.small_bytes % 16 != 0) return cudaErrorNotSupported;

  Params p;
  memset(&p, 0, sizeof(p));
  const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  cudaError_t e;
  // Boxes are sized for the padded widths; TMA zero-fills what lies beyond
  // the caller's tensors and clips stores to them.
  if ((e = encode_tmap_2d(&p.x_map, dt, 2, x, rows, Dt, BM, 64, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess) return e;
  if ((e = encode_tmap_2d(&p.out_map, dt, 2, out, rows, Ot, 32, 64, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return e;
  for (int l = 0; l < L; ++l) {
    const int K = l == 0 ? D : H;
    if ((e = encode_tmap_2d(&p.w_map[l], dt, 2, W[l], l == 0 ? Dt : Ht, layer_out(Ht, Ot, L, l), streamed ? 64 : K,
                            64, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
      return e;
    p.bias[l] = b != nullptr ? static_cast<const uint16_t*>(b[l]) : nullptr;
    p.nb[l] = layer_out(Ht, Ot, L, l);
  }
  p.store_h = h != nullptr && L > 1 ? 1 : 0;
  for (int l = 0; p.store_h && l < L - 1; ++l)
    if ((e = encode_tmap_2d(&p.h_map[l], dt, 2, h[l], rows, Ht, 32, 64, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
      return e;
  p.rows = static_cast<int>(rows);
  p.D = D;
  p.H = H;
  p.O = O;
  p.L = L;
  p.workers = E;
  p.cgroups = C;
  p.cshift = C == 4 ? 2 : C == 2 ? 1 : 0;
  p.mma_warps = nm;
  p.lo = lo;
  p.err = dev.err_word;

  void (*kernel)(Params);
  const bool square = O == H && !bf16;  // the pages' form gets its own instantiation
  const bool st = p.store_h != 0;
  // fp16 softplus chains carry their activations in log2 units (one
  // instruction fewer per pair on every layer before the last).  With
  // resident weights the unit changes are folded into the first and last
  // layers' weights (kFold), for any chain of two or more layers; with
  // streamed weights they cost one multiply per pair in those two layers,
  // which pays from four layers on.
  const bool log2u = act == kActSoftplus && !bf16 && !st && (L >= 4 || (L >= 2 && !streamed));
#define COALESCE_MLP_PICK(ACT)                                                                                 \
  kernel = bf16 ? (st ? mlp_fused_kernel<ACT, true, false, true> : mlp_fused_kernel<ACT, true, false, false>) \
               : square ? (st ? mlp_fused_kernel<ACT, false, true, true> : mlp_fused_kernel<ACT, false, true, false>) \
                        : (st ? mlp_fused_kernel<ACT, false, false, true> : mlp_fused_kernel<ACT, false, false, false>)
  switch (act) {
    case kActSoftplus:
      if (log2u && !streamed)
        kernel = square ? mlp_fused_kernel<kActSoftplus, false, true, false, true, true>
                        : mlp_fused_kernel<kActSoftplus, false, false, false, true, true>;
      else if (log2u)
        kernel = square ? mlp_fused_kernel<kActSoftplus, false, true, false, true>
                        : mlp_fused_kernel<kActSoftplus, false, false, false, true>;
      else
        COALESCE_MLP_PICK(kActSoftplus);
      break;
    case kActRelu:
      COALESCE_MLP_PICK(kActRelu);
      break;
    case kActGeluErf:
      COALESCE_MLP_PICK(kActGeluErf);
      break;
    default:
      COALESCE_MLP_PICK(kActNone);
      break;
  }
#undef COALESCE_MLP_PICK
  if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
    return e;
  const int64_t tiles = (rows + BM - 1) / BM;
  const int grid = static_cast<int>(tiles < dev.sm_count ? tiles : dev.sm_count);
  kernel<<<grid, 128 * C * E + 32 * nm + 32 + (WR > 0 ? 32 : 0), smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace coalesce
