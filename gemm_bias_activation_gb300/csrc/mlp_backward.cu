// Backward pass of the chained MLP in one persistent kernel (sm_103a).
//
// Layer l (0-based) maps a_l [rows, K_l] to z_l = a_l W_l + b_l [rows, N_l];
// a_0 = x, a_l = act(z_{l-1}) = h_{l-1} (stored by the training forward).
// Given g_{L-1} = dout = dLoss/dz_{L-1}, for l = L-1 .. 0:
//   db_l += sum over rows of g_l
//   dW_l += a_l^T g_l
//   g_{l-1} = (g_l W_l^T) * act'(a_l)        (l > 0; act' from the stored a_l)
//   dx = g_0 W_0^T                           (l = 0)
//
// The "MLP Megakernel" README ("Key ideas") runs the training backward as one
// fused kernel for small batches and, above 32K rows, as GEMMs for the weight
// gradients interleaved with the data-gradient computation.  On this GPU the
// fused form serves every batch size the shapes allow: each CTA keeps its own
// partial dW_l (fp32) in tensor memory across all of its row tiles, so the
// weight gradients need no pass of their own over the activations, and adds
// them into dW once at the end (TMA reduce-add).  Every row tile of dout, of
// each stored activation and of x is read once, dx is written once, and the
// data gradients g_l never leave the SM.
//
// Design (one CTA per SM, persistent over 128-row tiles, CTA-local tile t):
//   * All W_l stay in shared memory (one TMA load at the start, 64-column
//     blocks of K_l rows x 128 B, 128-B swizzle); row tiles go through a ring
//     of R slots of 128 rows x max width.  Tile t takes L + 1 consecutive ring
//     positions in the order the steps use them: dout, a_{L-1}, ..., a_0 = x.
//   * Step l of a tile reads G = g_l (the dout slot for l = L-1, otherwise the
//     slot of a_{l+1}, where step l+1 wrote g_l) and A = the slot of a_l.
//     The MMA warp issues, from one elected lane,
//       acc2 = G W_l^T     M = 128 rows, N = K_l, K = N_l; G K-major, W_l as
//                          stored is the K-major B operand of W_l^T
//     and commits it to acc_full, then
//       dW_l += A^T G      M = 128 (dW rows; A^T is A read MN-major, with rows
//                          K_l .. 127 taken from a zero block when K_l = 64),
//                          N = N_l, K = the tile's 128 rows; G read MN-major
//     and commits everything to dw_done and to the release of G's slot.  The
//     epilogue starts on acc2 while the dW MMAs run and writes over a_l (which
//     they read) only once dw_done has completed.
//     At a tile's first step the dW MMAs (G = dout) are issued before the
//     wait for the epilogue to release acc2.
//   * Epilogue warps (four lane quarters x C column groups) wait for
//     acc_full; warp (q, c) owns rows 32q .. 32q+31 (TMEM lanes) and a 1/C
//     share of the columns.  For l > 0 it reads acc2 (tcgen05.ld), multiplies
//     by act'(a_l) read from the A slot, rounds to the operand type and writes
//     g_{l-1} over a_l in place (the MMA reading a_l has completed).  For
//     l = 0 it writes dx into the x slot and stores it by TMA.
//   * Four column-sum warps add the columns of dout and of every g_{l-1}
//     over the tile's rows (db), each warp owning fixed 32-column blocks, in
//     fp32 shared-memory accumulators added into db once at the end; they run
//     beside the MMAs and the epilogue, off the chain between them.
//   * One I/O warp refills each slot as soon as its previous tile position is
//     released (by the MMA commit, every epilogue and every column-sum warp).
// Ragged row tails are zero-filled by TMA (zero rows add nothing) and the dx
// store is clipped.  Widths that are not multiples of 64 run rounded up to 64:
// the padded columns of dout, of every a_l and of W_l (and W_l's padded rows)
// load as zeros, so the padded columns of acc2 are 0, those of every g_l are
// 0 * act'(0) = 0, and the padded rows and columns of dW_l are 0; dW, db and
// dx are written only within the caller's extents.  Every wait is bounded; a wait that runs out records an
// error and its warp stops; the MMA warp drains its MMAs before TMEM is
// released.
#include "epilogue.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace coalesce {
namespace mlpbwd {

constexpr int BM = 128;
constexpr int kMaxLayers = 8;
constexpr int kMaxSlots = 16;
constexpr int kMaxGroups = 4;
constexpr int kSumWarps = 4;  // column-sum warps
constexpr int kMaxThreads = 32 * (4 * kMaxGroups + 2 + kSumWarps);
constexpr uint32_t kTileChunk = BM * 128u;  // one 64-column block of a row tile: 16 KiB
constexpr uint32_t kZeroBytes = 2048u;      // one k-step (16 rows x 128 B) of zeros
constexpr uint32_t kSmemLimit = 232448u;

__host__ __device__ inline uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }
__host__ __device__ inline int in_w(int D, int H, int l) { return l == 0 ? D : H; }
__host__ __device__ inline int out_w(int H, int O, int L, int l) { return l == L - 1 ? O : H; }

struct Layout {
  // relative to the start of dynamic shared memory
  uint32_t bar_off;  // w_full, acc_full, epi_done, drain, slot_full[R], slot_free[R], g_ready[R]
  uint32_t tmem_slot_off;
  uint32_t db_off;  // fp32 column sums, layer l's at db_idx[l]
  uint32_t small_bytes;
  // relative to the 1 KiB-aligned big base
  uint32_t w_off[kMaxLayers];
  uint32_t slot_off;
  uint32_t slot_bytes;
  uint32_t slots;     // R
  uint32_t zero_off;  // kZeroBytes of zeros (used when some K_l < 128)
  uint32_t big_bytes;
  uint32_t alloc_bytes;
  uint32_t db_idx[kMaxLayers];
  uint32_t db_count;
  uint32_t dw_col[kMaxLayers];  // TMEM column of dW_l (acc2 at column 0)
  uint32_t tmem_cols;
};

__host__ __device__ inline Layout make_layout(int D, int H, int O, int L, int R) {
  Layout lo{};
  uint32_t off = 0;
  lo.bar_off = off;
  off += 8u * (5u + 3u * static_cast<uint32_t>(R));
  lo.tmem_slot_off = off;
  off += 16;
  lo.db_off = align_up(off, 16);
  uint32_t ndb = 0;
  for (int l = 0; l < L; ++l) {
    lo.db_idx[l] = ndb;
    ndb += static_cast<uint32_t>(out_w(H, O, L, l));
  }
  lo.db_count = ndb;
  lo.small_bytes = align_up(lo.db_off + 4u * ndb, 16);
  uint32_t big = 0;
  int maxw = D > O ? D : O;
  if (L > 1 && H > maxw) maxw = H;
  int kmax = 0;
  bool need_zero = false;
  for (int l = 0; l < L; ++l) {
    const int K = in_w(D, H, l);
    lo.w_off[l] = big;
    big += static_cast<uint32_t>(out_w(H, O, L, l) / 64) * static_cast<uint32_t>(K) * 128u;
    kmax = K > kmax ? K : kmax;
    need_zero = need_zero || K < BM;
  }
  big = align_up(big, 1024);
  lo.slot_bytes = static_cast<uint32_t>(maxw / 64) * kTileChunk;
  lo.slot_off = big;
  lo.slots = static_cast<uint32_t>(R);
  big += static_cast<uint32_t>(R) * lo.slot_bytes;
  lo.zero_off = 0;
  if (need_zero) {
    lo.zero_off = big;
    big += kZeroBytes;
  }
  lo.big_bytes = big;
  // dynamic shared memory is at least 16-byte aligned: at most 1008 bytes of padding
  lo.alloc_bytes = lo.small_bytes + 1008u + big;
  uint32_t col = static_cast<uint32_t>(kmax);
  for (int l = 0; l < L; ++l) {
    col = align_up(col, 32);
    lo.dw_col[l] = col;
    col += static_cast<uint32_t>(out_w(H, O, L, l));
  }
  uint32_t cols = 32;
  while (cols < col) cols <<= 1;
  lo.tmem_cols = cols;
  return lo;
}

struct Params {
  CUtensorMap dout_map;            // dout [rows, O], box 128 x 64
  CUtensorMap a_map[kMaxLayers];   // a_0 = x [rows, D], a_l = h_{l-1} [rows, H]; box 128 x 64
  CUtensorMap w_map[kMaxLayers];   // W_l [K_l, N_l], box K_l x 64
  CUtensorMap dx_map;              // dx [rows, D], box 32 x 64 (store)
  CUtensorMap dw_map[kMaxLayers];  // dW_l fp32 [K_l, N_l], box 32 x 32 (reduce-add)
  float* db[kMaxLayers];           // fp32 [N_l] or nullptr
  Layout lo;
  int rows, D, H, O, L;  // widths rounded up to multiples of 64
  int Dt, Ht, Ot;        // the caller's widths (dW, db and dx extents)
  int cgroups;  // C
  int want_dx;
  uint32_t* err;
};

// A position in the slot ring: its slot and the parity of that slot's
// current use (positions advance one at a time, so no division is needed).
struct RingPos {
  int s;
  uint32_t ph;
  __device__ __forceinline__ void next(int R) {
    if (++s == R) {
      s = 0;
      ph ^= 1u;
    }
  }
};

// 8 columns of g = acc * act'(a): acc8 the fp32 accumulator values, av the
// 16-bit activations at the same positions; the result is rounded to 16 bits.
// (x0, x1) * s (one packed fp32 multiply).
__device__ __forceinline__ float2 mul2(float2 x, float s) {
  float2 r;
  asm("{\n\t.reg .b64 a, b, d;\n\t"
      "mov.b64 a, {%2, %3};\n\t"
      "mov.b64 b, {%4, %4};\n\t"
      "mul.rn.f32x2 d, a, b;\n\t"
      "mov.b64 {%0, %1}, d;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(x.x), "f"(x.y), "f"(s));
  return r;
}

// (g0, g1) = (a0, a1) * (1 - (t0, t1)), with one packed fma and one packed multiply.
__device__ __forceinline__ float2 mul_one_minus2(float2 a, float2 t) {
  float2 r;
  asm("{\n\t.reg .b64 ta, one, m1, d, av, g;\n\t"
      "mov.b64 ta, {%4, %5};\n\t"
      "mov.b64 one, {%6, %6};\n\t"
      "mov.b64 m1, {%7, %7};\n\t"
      "fma.rn.f32x2 d, ta, m1, one;\n\t"
      "mov.b64 av, {%2, %3};\n\t"
      "mul.rn.f32x2 g, av, d;\n\t"
      "mov.b64 {%0, %1}, g;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(t.x), "f"(t.y), "f"(1.0f), "f"(-1.0f));
  return r;
}

template <int kAct, bool kBf16>
__device__ __forceinline__ uint4 dact8(const uint32_t* acc8, uint4 av) {
  if constexpr (kAct == kActSoftplus) {
    // softplus' = 1 - e^-h = 1 - 2^(-h log2 e), two values at a time
    const uint32_t a[4] = {av.x, av.y, av.z, av.w};
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float2 h;
      if constexpr (kBf16) {
        h = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&a[k]));
      } else {
        h = __half22float2(*reinterpret_cast<const __half2*>(&a[k]));
      }
      const float2 e = mul2(h, -1.44269504088896341f);
      float2 t;
      asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(t.x) : "f"(e.x));
      asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(t.y) : "f"(e.y));
      const float2 g = mul_one_minus2(make_float2(__uint_as_float(acc8[2 * k]), __uint_as_float(acc8[2 * k + 1])), t);
      if constexpr (kBf16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(g.x, g.y);
        w[k] = *reinterpret_cast<uint32_t*>(&v);
      } else {
        w[k] = pack_f16x2(g.x, g.y);
      }
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
  const uint32_t a[4] = {av.x, av.y, av.z, av.w};
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float2 h;
    if constexpr (kBf16) {
      h = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&a[k]));
    } else {
      h = __half22float2(*reinterpret_cast<const __half2*>(&a[k]));
    }
    const float g0 = __uint_as_float(acc8[2 * k]) * dact_from_output<kAct>(h.x);
    const float g1 = __uint_as_float(acc8[2 * k + 1]) * dact_from_output<kAct>(h.y);
    if constexpr (kBf16) {
      __nv_bfloat162 v = __floats2bfloat162_rn(g0, g1);
      w[k] = *reinterpret_cast<uint32_t*>(&v);
    } else {
      w[k] = pack_f16x2(g0, g1);
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <bool kBf16>
__device__ __forceinline__ uint4 pack8(const uint32_t* acc8) {
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float v0 = __uint_as_float(acc8[2 * k]), v1 = __uint_as_float(acc8[2 * k + 1]);
    if constexpr (kBf16) {
      __nv_bfloat162 v = __floats2bfloat162_rn(v0, v1);
      w[k] = *reinterpret_cast<uint32_t*>(&v);
    } else {
      w[k] = pack_f16x2(v0, v1);
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Column sums over all 128 rows of a tile held in a slot (64-column blocks of
// 128 rows x 128 B, 16-byte chunk j of row r at j ^ (r & 7)), added into
// acc[col] (shared fp32).  Column-sum warp k takes the 32-column blocks
// k, k + kSumWarps, ...; in a block lane p = lane & 15 sums the column pair
// 2p, 2p+1 over half lane >> 4 of the rows, the halves walking their rows 4
// apart in the swizzle so that the 32 lanes hit 32 different banks.  Each
// column has one owner warp, so the update needs no atomic.
template <bool kBf16>
__device__ __forceinline__ void colsum_tile(const uint8_t* slot, int width, float* acc, uint32_t k, uint32_t lane) {
  const uint32_t half = lane >> 4;
  for (int cb = 32 * static_cast<int>(k); cb < width; cb += 32 * kSumWarps) {
    const int pc = cb + 2 * static_cast<int>(lane & 15u);
    const uint8_t* chunk = slot + static_cast<uint32_t>(pc / 64) * kTileChunk;
    const uint32_t unit = static_cast<uint32_t>(pc % 64) / 8u;
    const uint32_t within = static_cast<uint32_t>(pc % 8) * 2u;
    float s0 = 0.0f, s1 = 0.0f;
#pragma unroll 16
    for (uint32_t i = 0; i < 64; ++i) {
      const uint32_t r = 64u * half + ((i + 4u * half) & 63u);
      const uint32_t bits = *reinterpret_cast<const uint32_t*>(chunk + r * 128u + ((unit ^ (r & 7u)) << 4) + within);
      float2 v;
      if constexpr (kBf16) {
        v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bits));
      } else {
        v = __half22float2(*reinterpret_cast<const __half2*>(&bits));
      }
      s0 += v.x;
      s1 += v.y;
    }
    s0 += __shfl_xor_sync(0xffffffffu, s0, 16);
    s1 += __shfl_xor_sync(0xffffffffu, s1, 16);
    if (lane < 16) {
      acc[pc] += s0;
      acc[pc + 1] += s1;
    }
  }
}

// kLateA: the ring holds at most one tile's L + 1 positions, so the next
// tile's a_{L-1} is loaded late (its slot frees only after this tile's second
// step).  A tile's first acc2 then goes ahead of the wait for it, and its
// first dW MMAs after acc2 as at every other step.  Without it both operands
// of the first step are in early, and its dW MMAs go ahead of the wait for the
// epilogue instead.  (A compile-time choice: the issue loop's speed depends
// on its exact code.)
template <int kAct, bool kBf16, bool kLateA>
__global__ void __launch_bounds__(kMaxThreads, 1) mlp_backward_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const Layout& lo = p.lo;
  const int L = p.L;
  const int C = p.cgroups;
  const int R = static_cast<int>(lo.slots);
  const uint32_t nepi = 4u * static_cast<uint32_t>(C);
  const uint32_t sbase = smem_u32(smem_raw);
  const uint32_t base = (sbase + lo.small_bytes + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - sbase);
  float* db_s = reinterpret_cast<float*>(smem_raw + lo.db_off);
  const uint32_t warp = warp_index_uniform();
  const uint32_t lane = threadIdx.x % 32;
  const int num_tiles = (p.rows + BM - 1) / BM;
  const int my_tiles = (num_tiles - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                       static_cast<int>(gridDim.x);

  const uint32_t w_full = sbase + lo.bar_off;
  const uint32_t acc_full = w_full + 8u;
  const uint32_t epi_done = w_full + 16u;
  const uint32_t drain = w_full + 24u;
  auto slot_full = [&](int s) { return w_full + 32u + 8u * static_cast<uint32_t>(s); };
  auto slot_free = [&](int s) { return w_full + 32u + 8u * static_cast<uint32_t>(R + s); };
  auto g_ready = [&](int s) { return w_full + 32u + 8u * static_cast<uint32_t>(2 * R + s); };
  const uint32_t dw_done = w_full + 32u + 8u * static_cast<uint32_t>(3 * R);  // a step's dW MMAs have read a_l
  auto slot_addr = [&](int s) { return base + lo.slot_off + static_cast<uint32_t>(s) * lo.slot_bytes; };
  auto slot_ptr = [&](int s) { return gbase + lo.slot_off + static_cast<uint32_t>(s) * lo.slot_bytes; };
  auto tile_row = [&](int t) { return (static_cast<int>(blockIdx.x) + t * static_cast<int>(gridDim.x)) * BM; };

  // ---- set-up: barriers, TMEM, zeroed column sums and zero block, weights
  if (threadIdx.x == 0) {
    mbar_init(w_full, 1);
    mbar_init(acc_full, 1);
    mbar_init(epi_done, nepi);
    mbar_init(drain, 1);
    mbar_init(dw_done, 1);
    for (int s = 0; s < R; ++s) {
      mbar_init(slot_full(s), 1);
      // the MMA commit, every epilogue warp and every column-sum warp
      mbar_init(slot_free(s), 1u + nepi + static_cast<uint32_t>(kSumWarps));
      mbar_init(g_ready(s), nepi);  // once per use of the slot (see the epilogue)
    }
    fence_mbarrier_init();
  }
  if (warp == 0) {
    tmem_alloc(sbase + lo.tmem_slot_off, lo.tmem_cols);
    tmem_relinquish_alloc_permit();
  }
  for (uint32_t i = threadIdx.x; i < lo.db_count; i += blockDim.x) db_s[i] = 0.0f;
  if (lo.zero_off != 0)
    for (uint32_t i = threadIdx.x; i < kZeroBytes / 16u; i += blockDim.x)
      *reinterpret_cast<uint4*>(gbase + lo.zero_off + 16u * i) = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();  // the zero block is read by the MMA (async proxy)
  __syncthreads();
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&p.dout_map);
    uint32_t wbytes = 0;
    for (int l = 0; l < L; ++l)
      wbytes += static_cast<uint32_t>(out_w(p.H, p.O, L, l) / 64) * static_cast<uint32_t>(in_w(p.D, p.H, l)) * 128u;
    mbar_arrive_expect_tx(w_full, wbytes);
    for (int l = 0; l < L; ++l) {
      const int K = in_w(p.D, p.H, l);
      for (int j = 0; j < out_w(p.H, p.O, L, l) / 64; ++j)
        tma_load_2d(base + lo.w_off[l] + static_cast<uint32_t>(j * K) * 128u, &p.w_map[l], w_full, j * 64, 0);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(smem_raw + lo.tmem_slot_off);

  if (warp == nepi + 1) {
    // ---------------------------------------------------------------- I/O: slot refills
    if (lane == 0) {
      bool ok = true;
      RingPos c{0, 0u};
      bool wrapped = false;  // every slot has been used once
      for (int t = 0; ok && t < my_tiles; ++t) {
        const int row0 = tile_row(t);
        for (int j = 0; j <= L; ++j, c.next(R)) {
          const int s = c.s;
          if (s == 0 && (t > 0 || j > 0)) wrapped = true;
          if (wrapped && !mbar_wait(slot_free(s), c.ph ^ 1u, p.err, kErrWaitMlpBackward)) {
            ok = false;
            break;
          }
          const CUtensorMap* map = j == 0 ? &p.dout_map : &p.a_map[L - j];
          const int width = j == 0 ? p.O : in_w(p.D, p.H, L - j);
          mbar_arrive_expect_tx(slot_full(s), static_cast<uint32_t>(width / 64) * kTileChunk);
          for (int c = 0; c < width / 64; ++c)
            tma_load_2d(slot_addr(s) + static_cast<uint32_t>(c) * kTileChunk, map, slot_full(s), c * 64, row0);
        }
      }
    }
    __syncwarp();
  } else if (warp == nepi) {
    // ---------------------------------------------------------------- MMA issuer
    bool ok = mbar_wait(w_full, 0, p.err, kErrWaitMlpBackward);
    uint32_t step = 0;
    RingPos cg{0, 0u};  // ring position of G (the tile's dout at its first step)
    for (int t = 0; ok && t < my_tiles; ++t, cg.next(R)) {  // the extra advance skips the x position
      for (int l = L - 1; ok && l >= 0; --l, cg.next(R)) {
        RingPos ca = cg;
        ca.next(R);
        const int sg = cg.s, sa = ca.s;
        const int K = in_w(p.D, p.H, l);
        const int N = out_w(p.H, p.O, L, l);
        if constexpr (kLateA) {
          // a tile's first step: G (dout) now, its A tile only before the dW MMAs
          if (l == L - 1) ok = mbar_wait_warp(slot_full(sg), cg.ph, p.err, kErrWaitMlpBackward);
          else ok = mbar_wait_warp(slot_full(sa), ca.ph, p.err, kErrWaitMlpBackward);
        } else {
          if (l == L - 1) ok = mbar_wait_warp(slot_full(sg), cg.ph, p.err, kErrWaitMlpBackward);
          if (ok) ok = mbar_wait_warp(slot_full(sa), ca.ph, p.err, kErrWaitMlpBackward);
        }
        if (!ok) break;
        const uint32_t g_addr = slot_addr(sg);
        const uint32_t a_addr = slot_addr(sa);
        // dW_l += A^T G (both MN-major; k-step = 16 tile rows = 2048 B)
        auto issue_dw = [&]() {
          const uint32_t idesc1 = idesc_f16_f32acc(kBf16, true, true, BM, static_cast<uint32_t>(N));
          for (int ks = 0; ks < BM / 16; ++ks) {
            const uint32_t a_start = a_addr + static_cast<uint32_t>(ks) * 2048u;
            const uint32_t lbo_a = K >= BM ? kTileChunk : base + lo.zero_off - a_start;
            const uint64_t ad = smem_desc_sw128(a_start, lbo_a, 1024);
            const uint64_t bd = smem_desc_sw128(g_addr + static_cast<uint32_t>(ks) * 2048u, kTileChunk, 1024);
            tc_mma_f16(tmem_base + lo.dw_col[l], ad, bd, idesc1, (t > 0 || ks > 0) ? 1u : 0u);
          }
        };
        // At a tile's first step G is dout, already loaded: its dW MMAs need
        // nothing from the epilogue and go ahead of the wait for it.
        if (!kLateA && l == L - 1) {
          tc_fence_after_sync();
          if (elect_one()) issue_dw();
          __syncwarp();
        }
        // acc2 has been read and (l < L-1) g_l written by the previous step
        if (step > 0) ok = mbar_wait_warp(epi_done, (step - 1u) & 1u, p.err, kErrWaitMlpBackward);
        if (!ok) break;
        tc_fence_after_sync();
        if (elect_one()) {
          if (l > 0 || p.want_dx) {
            // acc2 = G W_l^T
            const uint32_t idesc = idesc_f16_f32acc(kBf16, false, false, BM, static_cast<uint32_t>(K));
            const uint64_t ad0 = smem_desc_sw128(g_addr, 16, 1024);
            const uint64_t bd0 = smem_desc_sw128(base + lo.w_off[l], 16, 1024);
            for (int ks = 0; ks < N / 16; ++ks) {
              const uint64_t ad = ad0 + static_cast<uint64_t>(((ks / 4) * kTileChunk + (ks % 4) * 32) >> 4);
              const uint64_t bd = bd0 + static_cast<uint64_t>(((ks / 4) * K * 128 + (ks % 4) * 32) >> 4);
              tc_mma_f16(tmem_base, ad, bd, idesc, ks > 0 ? 1u : 0u);
            }
          }
          tc_commit(acc_full);
          if constexpr (!kLateA) {
            // dW_l after acc2, so that the epilogue can start on acc2 while the
            // dW MMAs run; it overwrites a_l (which they read) only after dw_done.
            if (l < L - 1) issue_dw();
            tc_commit(dw_done);
            tc_commit(slot_free(sg));
            if (l == 0) tc_commit(slot_free(sa));
          }
        }
        __syncwarp();
        if constexpr (kLateA) {
          if (l == L - 1) {
            ok = mbar_wait_warp(slot_full(sa), ca.ph, p.err, kErrWaitMlpBackward);
            if (!ok) break;
            tc_fence_after_sync();
          }
          if (elect_one()) {
            // dW_l after acc2 (see above)
            issue_dw();
            tc_commit(dw_done);
            tc_commit(slot_free(sg));
            if (l == 0) tc_commit(slot_free(sa));
          }
          __syncwarp();
        }
        ++step;
      }
    }
    // Every MMA issued above has completed before TMEM can be released.
    if (elect_one()) tc_commit(drain);
    __syncwarp();
    mbar_wait(drain, 0, p.err, kErrWaitMlpBackward);
  } else if (warp < nepi) {
    // ---------------------------------------------------------------- epilogue warps
    const uint32_t q = warp & 3u;
    const int cg = static_cast<int>(warp >> 2);
    const uint32_t row = 32u * q + lane;
    const uint32_t row_sw = row & 7u;
    const uint32_t lane_base = (32u * q) << 16;
    const uint32_t leader = lane == 0 ? 1u : 0u;
    uint32_t step = 0;
    int pend = -1;  // x slot whose dx store has not yet been seen to read it
    bool ok = true;
    RingPos cgp{0, 0u};  // ring position of G
    for (int t = 0; ok && t < my_tiles; ++t, cgp.next(R)) {  // the extra advance skips the x position
      for (int l = L - 1; ok && l >= 0; --l, cgp.next(R)) {
        RingPos ca = cgp;
        ca.next(R);
        const int sg = cgp.s, sa = ca.s;
        const int K = in_w(p.D, p.H, l);
        // the A tile was written by TMA: observe its load too
        if (!mbar_wait_warp(acc_full, step & 1u, p.err, kErrWaitMlpBackward) ||
            !mbar_wait_warp(slot_full(sa), ca.ph, p.err, kErrWaitMlpBackward)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        if (pend >= 0) {
          bulk_read_done_arrive_if(slot_free(pend), leader);
          pend = -1;
        }
        uint8_t* as = slot_ptr(sa);
        if (l > 0) {
          // g_{l-1} = acc2 * act'(a_l), over a_l in place; 32 accumulator
          // columns per TMEM load
          const int kc = K / C;
          const int c_lo = cg * kc;
          if (kc == 32) {
            // one 32-column block: g into registers while dW_l may still read
            // a_l, then written over a_l once it has
            uint32_t acc[32];
            tmem_ld_32x32b_x32(tmem_base + lane_base + static_cast<uint32_t>(c_lo), acc);
            tmem_ld_wait();
            uint8_t* rowp = as + static_cast<uint32_t>(c_lo / 64) * kTileChunk + row * 128u;
            const uint32_t j0 = static_cast<uint32_t>(c_lo % 64) / 8u;
            uint4 gv[4];
#pragma unroll
            for (uint32_t j = 0; j < 4; ++j)
              gv[j] = dact8<kAct, kBf16>(acc + 8 * j, *reinterpret_cast<const uint4*>(rowp + (((j0 + j) ^ row_sw) << 4)));
            if (!mbar_wait_warp(dw_done, step & 1u, p.err, kErrWaitMlpBackward)) {
              ok = false;
              break;
            }
#pragma unroll
            for (uint32_t j = 0; j < 4; ++j) *reinterpret_cast<uint4*>(rowp + (((j0 + j) ^ row_sw) << 4)) = gv[j];
          } else {
            if (!mbar_wait_warp(dw_done, step & 1u, p.err, kErrWaitMlpBackward)) {
              ok = false;
              break;
            }
            for (int c0 = c_lo; c0 < c_lo + kc; c0 += 32) {
              uint32_t acc[32];
              tmem_ld_32x32b_x32(tmem_base + lane_base + static_cast<uint32_t>(c0), acc);
              tmem_ld_wait();
              uint8_t* rowp = as + static_cast<uint32_t>(c0 / 64) * kTileChunk + row * 128u;
              const uint32_t j0 = static_cast<uint32_t>(c0 % 64) / 8u;
#pragma unroll
              for (uint32_t j = 0; j < 4; ++j) {
                uint4* ptr = reinterpret_cast<uint4*>(rowp + (((j0 + j) ^ row_sw) << 4));
                *ptr = dact8<kAct, kBf16>(acc + 8 * j, *ptr);
              }
            }
          }
          fence_proxy_async_smem();  // the next step's MMA reads what was written
          __syncwarp();
        } else if (p.want_dx) {
          // the dW_0 MMAs read x from this slot: dx goes there only after them
          if (!mbar_wait_warp(dw_done, step & 1u, p.err, kErrWaitMlpBackward)) {
            ok = false;
            break;
          }
          // dx into the x slot, out in 32-row x 64-column boxes, each written
          // and stored by one warp (with 32-column shares the other warps of
          // a quarter sit this step out)
          const int dcw = p.D / C >= 64 ? p.D / C : 64;
          const int c_lo = cg * dcw;
          if (c_lo < p.D) {
            for (int c0 = c_lo; c0 < c_lo + dcw; c0 += 64) {
              uint32_t acc[64];
              tmem_ld_32x32b_x32(tmem_base + lane_base + static_cast<uint32_t>(c0), acc);
              tmem_ld_32x32b_x32(tmem_base + lane_base + static_cast<uint32_t>(c0 + 32), acc + 32);
              tmem_ld_wait();
              uint8_t* rowp = as + static_cast<uint32_t>(c0 / 64) * kTileChunk + row * 128u;
#pragma unroll
              for (uint32_t j = 0; j < 8; ++j)
                *reinterpret_cast<uint4*>(rowp + ((j ^ row_sw) << 4)) = pack8<kBf16>(acc + 8 * j);
            }
            fence_proxy_async_smem();  // the dx store reads what was written
            __syncwarp();
            for (int c = c_lo; c < c_lo + dcw; c += 64)
              tma_store_2d_if(&p.dx_map, slot_addr(sa) + static_cast<uint32_t>(c / 64) * kTileChunk + 32u * q * 128u,
                              c, tile_row(t) + static_cast<int>(32u * q), leader);
            bulk_commit_group_if(leader);
            // With three or more slots the release waits for the next step
            // (the next tile's first step never needs this slot); with two,
            // the next tile's second load goes here, so release it now.
            if (R < 3) bulk_wait_group_read_if(leader);
            __syncwarp();
            if (R >= 3) pend = sa;
          }
        }
        tc_fence_before_sync();
        __syncwarp();
        mbar_arrive_if(epi_done, leader);
        mbar_arrive_if(slot_free(sg), leader);
        // One g_ready phase per use of a slot: dout's at step L-1, and every
        // A slot's at its step (for l > 0 after g_{l-1} is written there).
        if (l == L - 1) mbar_arrive_if(g_ready(sg), leader);
        mbar_arrive_if(g_ready(sa), leader);
        if (l == 0 && pend < 0) mbar_arrive_if(slot_free(sa), leader);
        ++step;
      }
    }
    // ---- end: every dx store done, then this CTA's dW and db go out
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
    // no epilogue or column-sum warp still reads a slot: they become staging buffers
    named_barrier_sync(1, (nepi + static_cast<uint32_t>(kSumWarps)) * 32u);
    {
      // two 32 x 32 fp32 staging boxes (128-B swizzle) per warp
      const uint32_t stage = base + lo.slot_off + warp * 8192u;
      uint8_t* stage_p = gbase + lo.slot_off + warp * 8192u;
      uint32_t buf = 0;
      for (int l = 0; l < L; ++l) {
        const int Kt = in_w(p.Dt, p.Ht, l);        // the caller's dW_l is [Kt, Nt]
        const int Nt = out_w(p.Ht, p.Ot, L, l);
        const int nc = out_w(p.H, p.O, L, l) / C;
        if (static_cast<int>(32u * q) >= Kt) continue;  // rows of dW beyond K_l
        for (int c0 = cg * nc; c0 < (cg + 1) * nc && c0 < Nt; c0 += 32) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tmem_base + lane_base + lo.dw_col[l] + static_cast<uint32_t>(c0), r);
          tmem_ld_wait();
          if (lane == 0) bulk_wait_group_read<1>();  // the store from this buffer two boxes ago has read it
          __syncwarp();
          uint8_t* rowp = stage_p + buf * 4096u + lane * 128u;
#pragma unroll
          for (uint32_t j = 0; j < 8; ++j)
            *reinterpret_cast<uint4*>(rowp + ((j ^ (lane & 7u)) << 4)) =
                make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_reduce_add_2d(&p.dw_map[l], stage + buf * 4096u, c0, static_cast<int>(32u * q));
            bulk_commit_group();
          }
          buf ^= 1u;
        }
      }
      if (lane == 0) bulk_wait_group<0>();
      __syncwarp();
    }
  } else {
    // ---------------------------------------------------------------- column sums (db)
    // Warp k sums its 32-column blocks of dout (db_{L-1}) once loaded, and of
    // each g_{l-1} once the epilogue has written it (g_ready), over all 128
    // rows, while the tensor cores and the epilogue go on; it releases each
    // slot use like the other consumers.
    const uint32_t k = warp - (nepi + 2u);
    bool ok = true;
    RingPos c{0, 0u};
    for (int t = 0; ok && t < my_tiles; ++t) {
      for (int j = 0; j <= L; ++j, c.next(R)) {
        const int s = c.s;
        const uint32_t par = c.ph;
        if (!mbar_wait_warp((j == 0 || j == L) ? slot_full(s) : g_ready(s), par, p.err, kErrWaitMlpBackward)) {
          ok = false;
          break;
        }
        if (j == 0) {
          if (p.db[L - 1] != nullptr) colsum_tile<kBf16>(slot_ptr(s), p.O, db_s + lo.db_idx[L - 1], k, lane);
        } else if (j < L) {
          const int l = L - j;  // the slot held a_l and now holds g_{l-1}
          if (p.db[l - 1] != nullptr) colsum_tile<kBf16>(slot_ptr(s), p.H, db_s + lo.db_idx[l - 1], k, lane);
        }
        __syncwarp();
        mbar_arrive_if(slot_free(s), lane == 0 ? 1u : 0u);
      }
    }
    named_barrier_sync(1, (nepi + static_cast<uint32_t>(kSumWarps)) * 32u);  // slots free for staging
    // this warp's columns of every db_l
    for (int l = 0; l < L; ++l) {
      if (p.db[l] == nullptr) continue;
      const int W = out_w(p.Ht, p.Ot, L, l);  // the caller's width (a multiple of 8)
      for (int cb = 32 * static_cast<int>(k); cb < W; cb += 32 * kSumWarps) {
        if (lane < 16 && cb + 2 * static_cast<int>(lane) < W) {
          const int pc = cb + 2 * static_cast<int>(lane);
          atomicAdd(p.db[l] + pc, db_s[lo.db_idx[l] + static_cast<uint32_t>(pc)]);
          atomicAdd(p.db[l] + pc + 1, db_s[lo.db_idx[l] + static_cast<uint32_t>(pc) + 1u]);
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, lo.tmem_cols);
  }
}

// The shapes this kernel implements, in the padded widths it runs on: every
// width a multiple of 64, K_l <= 128 (dW_l fits one 128-lane accumulator),
// N_l <= 256, acc2 and every dW_l within 512 TMEM columns, the weights and at
// least two slots in shared memory.
bool plan(int D, int H, int O, int L, Layout* lo_out, int* c_out) {
  if (L < 1 || L > kMaxLayers) return false;
  for (int l = 0; l < L; ++l) {
    const int K = in_w(D, H, l), N = out_w(H, O, L, l);
    if (K % 64 != 0 || N % 64 != 0 || K > BM || N > 256) return false;
  }
  int R = 0;
  Layout lo{};
  for (int r = kMaxSlots; r >= 2; --r) {
    lo = make_layout(D, H, O, L, r);
    if (lo.alloc_bytes <= kSmemLimit) {
      R = r;
      break;
    }
  }
  if (R == 0 || lo.tmem_cols > 512) return false;
  // Column groups: every per-warp share of a width (K_l for acc2 and dx,
  // N_l for the dW write-back) whole 32-column blocks, and two 4 KiB staging
  // boxes per epilogue warp within the slots.
  int C = kMaxGroups;
  for (int l = 0; l < L; ++l) {
    while (C > 1 && (in_w(D, H, l) % (32 * C) != 0 || out_w(H, O, L, l) % (32 * C) != 0)) C /= 2;
  }
  while (C > 1 && static_cast<uint64_t>(4 * C) * 8192u > static_cast<uint64_t>(lo.slots) * lo.slot_bytes) C /= 2;
  *lo_out = lo;
  *c_out = C;
  return true;
}

}  // namespace mlpbwd

static inline int pad64(int64_t w) { return static_cast<int>((w + 63) / 64 * 64); }

bool mlp_backward_fused_supported(int64_t D, int64_t H, int64_t O, int L) {
  mlpbwd::Layout lo;
  int C;
  return D >= 1 && H >= 1 && O >= 1 && D % 8 == 0 && H % 8 == 0 && O % 8 == 0 && D <= 256 && H <= 256 &&
         O <= 256 && mlpbwd::plan(pad64(D), pad64(H), pad64(O), L, &lo, &C);
}

cudaError_t launch_mlp_backward_fused(const DeviceCtx& dev, int64_t rows, int Dt, int Ht, int Ot, int L, bool bf16,
                                      const void* x, const void* const* W, const void* const* h, const void* dout,
                                      void* dx, float* const* dW, float* const* db, int act, cudaStream_t stream) {
  using namespace mlpbwd;
  // The tensor maps take the caller's widths (multiples of 8); the kernel's
  // layout takes them rounded up to 64, the padding zero-filled on load.
  if (!mlp_backward_fused_supported(Dt, Ht, Ot, L)) return cudaErrorNotSupported;
  const int D = pad64(Dt), H = pad64(Ht), O = pad64(Ot);
  Layout lo;
  int C;
  if (!plan(D, H, O, L, &lo, &C)) return cudaErrorNotSupported;
  static_assert(sizeof(Params) <= 4096, "kernel parameters exceed 4 KiB");
  Params p;
  memset(&p, 0, sizeof(p));
  const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  cudaError_t e;
  if ((e = encode_tmap_2d(&p.dout_map, dt, 2, dout, rows, Ot, BM, 64, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
    return e;
  for (int l = 0; l < L; ++l) {
    const int K = in_w(D, H, l);
    const int Kt = in_w(Dt, Ht, l), Nt = out_w(Ht, Ot, L, l);
    const void* a = l == 0 ? x : h[l - 1];
    if ((e = encode_tmap_2d(&p.a_map[l], dt, 2, a, rows, Kt, BM, 64, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
      return e;
    if ((e = encode_tmap_2d(&p.w_map[l], dt, 2, W[l], Kt, Nt, K, 64, CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
      return e;
    if ((e = encode_tmap_2d(&p.dw_map[l], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dW[l], Kt, Nt, 32, 32,
                            CU_TENSOR_MAP_SWIZZLE_128B)) != cudaSuccess)
      return e;
    p.db[l] = db != nullptr ? db[l] : nullptr;
    if ((e = cudaMemsetAsync(dW[l], 0, sizeof(float) * Kt * Nt, stream)) != cudaSuccess) return e;
    if (p.db[l] != nullptr && (e = cudaMemsetAsync(p.db[l], 0, sizeof(float) * Nt, stream)) != cudaSuccess) return e;
  }
  p.want_dx = dx != nullptr ? 1 : 0;
  if ((e = encode_tmap_2d(&p.dx_map, dt, 2, dx != nullptr ? dx : x, rows, Dt, 32, 64, CU_TENSOR_MAP_SWIZZLE_128B)) !=
      cudaSuccess)
    return e;
  p.lo = lo;
  p.rows = static_cast<int>(rows);
  p.D = D;
  p.H = H;
  p.O = O;
  p.Dt = Dt;
  p.Ht = Ht;
  p.Ot = Ot;
  p.L = L;
  p.cgroups = C;
  p.err = dev.err_word;

  void (*kernel)(Params);
  switch (act) {
    case kActSoftplus:
      // the softplus chain (the pages' training form) gets the late-A order
      // when its ring holds one tile; the other activations keep the default
      if (static_cast<int>(lo.slots) <= L + 1)
        kernel = bf16 ? mlp_backward_kernel<kActSoftplus, true, true> : mlp_backward_kernel<kActSoftplus, false, true>;
      else
        kernel = bf16 ? mlp_backward_kernel<kActSoftplus, true, false> : mlp_backward_kernel<kActSoftplus, false, false>;
      break;
    case kActRelu:
      kernel = bf16 ? mlp_backward_kernel<kActRelu, true, false> : mlp_backward_kernel<kActRelu, false, false>;
      break;
    default:
      kernel = bf16 ? mlp_backward_kernel<kActNone, true, false> : mlp_backward_kernel<kActNone, false, false>;
      break;
  }
  if ((e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, lo.alloc_bytes)) != cudaSuccess)
    return e;
  const int64_t tiles = (rows + BM - 1) / BM;
  const int grid = static_cast<int>(tiles < dev.sm_count ? tiles : dev.sm_count);
  kernel<<<grid, 32 * (4 * C + 2 + kSumWarps), lo.alloc_bytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace coalesce
