// FP32 SGEMM on the CUDA cores: C = alpha * op(A) * op(B) + beta * C.
//
// What the pages contribute (design ideas, not code):
//  - "Optimizing GEMM on Apple's M5 from scratch, Part 1": shared-memory
//    tiling ("Kernels 2 and 3: Shared Memory Tiling": every input tile is
//    loaded once per block and reused by all its threads) and thread
//    coarsening ("Kernel 4: 1D Thread Coarsening": one thread owns several
//    outputs so an operand value held in a register feeds several FMAs).  Here
//    the coarsening is two-dimensional, an 8 x 8 register block per thread, the
//    register blocking of "From a C loop to a GPU kernel" ("One thread, four
//    outputs", 2x2 there, with 4x4 and 8x8 named as the next steps).
//  - "From a C loop to a GPU kernel", "The bubble between tiles": the next K
//    tile is fetched while the current one is consumed.  Here a 3-stage
//    cp.async ring.
//  - "Metal GEMM Kernels for LoRA Training", section 3: the transposed
//    operand cost instruction count, not memory traffic.  Here no operand is
//    transposed in memory at all: each operand is staged in the orientation it
//    is stored in, and the inner loop reads it with 128-bit shared loads along
//    whichever dimension is contiguous (k for A[M,K] / B[N,K]; m or n for
//    A[K,M] / B[K,N]).
//  - "Part 1", "Kernel 1: Naive Implementation" (and "Coalescing" in the C-loop
//    post): consecutive threads own consecutive columns, so global loads are
//    coalesced; here every global load is a 16-byte cp.async and a warp's loads
//    cover whole 64- or 512-byte row segments.
//
// Tile: (64 * WARPS_M) x (4 * LN * WARPS_N) outputs per block (warps of
// 64 x 4 LN, each lane 8 x LN outputs split into 4-wide groups): 128 x 128 at
// K step 64, one block per SM, in general; 256 x 32 at K step 32, two blocks
// per SM, for N <= 32; 128 x 256 (LN = 16) and 128 x 64 as opt-in shapes.
// This header is instantiated once per tile shape, each in its own
// translation unit.
//
// Two kernels share the inner product and the epilogue: sgemm_ffma_kernel,
// whose warps stage every layout themselves with cp.async copies and a block
// barrier per K step, and sgemm_ws_kernel, for operands stored k-major with
// aligned rows (what the packing pre-pass writes), where a producer warp
// feeds the ring by TMA and the math warps synchronise only through the
// stages' mbarriers (measured at 4096^3: 2.22 -> 1.92 ms, the FMA pipe 80 ->
// 90 % busy).  The inner product runs on Blackwell's
// paired FP32 FMA (fma.rn.f32x2): one instruction updates two adjacent outputs
// of a lane, halving the issue slots the FMAs take (the scalar-FMA version of
// this kernel was bound by instruction issue).  Each half of the pair is an
// IEEE fp32 FMA (round to nearest even); no fast-math, denormals kept.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"
#include "tensor_map.h"

namespace gb300 {
namespace {

#ifndef GB300_SG_STAGES
#define GB300_SG_STAGES 3
#endif
constexpr int STAGES = GB300_SG_STAGES;
// Block tile: (64 * WM) x (4 * LN * WN) outputs, WM x WN warps of 64 x 4 LN
// (each lane 8 rows x LN columns, LN = 8 or 16), K step BK_, NST-stage ring,
// sized for MINB resident blocks per SM.
template <int WM, int WN, int BK_, int MINB, int LN_ = 8, int NST = STAGES>
struct Tile {
  static constexpr int WARPS_M = WM, WARPS_N = WN;
  static constexpr int LN = LN_;         // columns a lane owns
  static constexpr int JP = LN / 2;      // ... as column pairs
  static constexpr int HB = LN / 4;      // ... as 4-column groups, 16 columns apart
  static constexpr int WARP_N = 4 * LN;  // columns a warp owns
  static constexpr int BM = 64 * WM, BN = WARP_N * WN, BK = BK_;
  static constexpr int NSTAGES = NST;
  static constexpr int THREADS = 32 * WM * WN;
  static constexpr int MIN_BLOCKS = MINB;
  static constexpr int APAD = BM + 4;  // k-major tile rows padded: conflict-free transposing writes
  static constexpr int BPAD = BN + 4;
  static constexpr int A_FLOATS = (BM * BK > BK * APAD) ? BM * BK : BK * APAD;
  static constexpr int B_FLOATS = BK * BPAD;
  static constexpr int STAGE_FLOATS = A_FLOATS + B_FLOATS;
  static constexpr int SMEM_BYTES = NSTAGES * STAGE_FLOATS * 4;
  // chunk permutation within a row tile row (BK/4 chunks): XOR with (row / 4)
  // modulo the chunk count, at most 8
  static constexpr int SWZ_MASK = (BK / 4 < 8 ? BK / 4 : 8) - 1;
  static_assert(BK == 16 || BK == 32 || BK == 64, "K step");
  static_assert(LN == 8 || LN == 16, "lane columns");
  static_assert(NSTAGES >= 2, "stages");
};
// the general tile (128 x 128 at the defaults: 195 KiB at BK 64, 3 stages) and
// the narrow one for N <= 32 (256 x 32, BK 32, two blocks per SM)
using TileWide = Tile<SG_WARPS_M, SG_BN / 32, SG_BK, SG_BLOCKS_PER_SM>;
using TileNarrow = Tile<SGN_BM / 64, SGN_BN / 32, SGN_BK, SGN_BLOCKS_PER_SM, 8, SGN_STAGES>;
using TileBig = Tile<SGB_BM / 64, SGB_BN / 64, SGB_BK, 1, 16, SGB_STAGES>;
using TileHalf = Tile<SGH_BM / 64, SGH_BN / 32, SGH_BK, SGH_BLOCKS_PER_SM, 8, SGH_STAGES>;
static_assert(TileWide::BM == SG_BM && TileWide::BN == SG_BN, "tile shape");
static_assert(TileNarrow::BM == SGN_BM && TileNarrow::BN == SGN_BN, "tile shape");
static_assert(TileBig::BM == SGB_BM && TileBig::BN == SGB_BN, "tile shape");
static_assert(TileHalf::BM == SGH_BM && TileHalf::BN == SGH_BN, "tile shape");

// Tile rasterisation: blocks walk GROUP tile-rows column by column, so each B
// panel is fetched from DRAM once per group while the group's A panels stay in
// L2.  The host picks GROUP so those A panels take about a quarter of L2
// (32 MB): measured at 4096^3, 8-row groups read 352 MB from DRAM, 16-row
// groups (the pick there) 334-336 MB and 32-row groups (64 MB of A panels)
// 520 MB -- the L2 is split between the two dies.  (Even at 16 rows an A
// panel's K slice comes back one wave of 152 tiles later, after ~61 MB of
// other slices, and is read again.)
constexpr int64_t RASTER_L2_BYTES = 32ll << 20;

// Compile-time tuning knobs (measured on GB300 at 4096^3; the defaults won;
// K step and stage count are GB300_SG_BK in internal.h and GB300_SG_STAGES:
// with cp.async staging 64 x 3 beat 32 x 3, 32 x 4, 64 x 2 and 16 x 6 by
// 0.4-5 %, and with TMA staging 32 x 6 was 2.5 % slower (1.968 against 1.919
// ms; 8192^3 3 %); 128 x 64 tiles at two blocks per SM (GB300_SG_BN=64,
// GB300_SG_MIN_BLOCKS=2) were 1-3 % slower; loading the next K step's
// fragments into a second register set gained nothing; unrolling the whole
// 16-chunk loop (GB300_SG_KC_UNROLL=16) was level at 4096^3 and up to 6 %
// slower on short K):
//  GB300_SG_MIN_BLOCKS  blocks per SM the register budget is sized for
//  GB300_SG_KC_UNROLL   unrolling of the 4-k chunk loop
#ifndef GB300_SG_KC_UNROLL
#define GB300_SG_KC_UNROLL 8
#endif
constexpr int KC_UNROLL = GB300_SG_KC_UNROLL;

struct Params {
  const float* A;
  const float* B;
  float* C;
  float* partial;
  int64_t lda, ldb, ldc;
  int M, N, K;
  int k_slice;
  int tiles_m, tiles_n;
  int group_m;  // tile-rows per rasterisation group
  float alpha, beta;
  // strided batch: blockIdx.y selects matrices A + y*stride_a, B + y*stride_b,
  // C + y*stride_c (all zero for a single GEMM)
  int64_t stride_a, stride_b, stride_c;
  // persistent launches (KIND_PERSIST): gridDim.x blocks first take whole
  // tiles t = blockIdx.x + i * gridDim.x below dp_tiles, then share the
  // remaining tiles' K steps evenly (block b owns steps [b*I/G, (b+1)*I/G) of
  // the I = sk_iters steps, G = gridDim.x, tiles in order, kiters steps
  // each).  A tile cut between blocks is finished by the last block to
  // arrive: partials in sk_ws[block][slot], arrivals counted in sk_cnt.
  int dp_tiles, kiters;
  int64_t sk_iters;
  float* sk_ws;
  unsigned int* sk_cnt;
  Epilogue ep;  // bias (fp32, per column) and activation, applied before the store
  int c_vec;    // C rows (and batch entries) 16-byte aligned: float4 epilogue accesses
  // warp-specialised variant: the device status word its bounded waits flag
  // their expiry in, their limit, and a test hook (1: the first stage's loads
  // are never issued, so the first wait expires)
  unsigned int* status;
  uint64_t timeout_ns;
  int fault_injection;
};

// Kernel kinds: one output tile per block (C), one K slice of a tile per
// block (raw partials, reduced by a second kernel), or persistent blocks over
// whole tiles and then shared K steps (C, with in-kernel fix-up).
constexpr int KIND_TILE = 0, KIND_SPLIT = 1, KIND_PERSIST = 2;

// ---------------------------------------------------------------- staging
// Tile layouts per operand and stage:
//  "k-major" tile : 32 rows (k) x BM or BN (m or n), rows padded by 4 floats.
//                   An operand stored with m/n contiguous (A[K,M], B[K,N]) is
//                   copied row by row with 16-byte copies.  B stored [N,K] is
//                   transposed into it on the way in with 4-byte copies -- the
//                   transposing write of "Metal GEMM Kernels for LoRA Training",
//                   section 3, done by the async-copy unit: a warp reads 4 rows
//                   x 32 bytes of global memory and, thanks to the padding,
//                   writes 32 distinct banks.  B must be k-major because the
//                   paired FMA needs column pairs (n, n+1) in adjacent registers.
//  "row" tile     : BM rows (m) x 32 k, 128-byte rows whose eight 16-byte chunks
//                   are permuted by chunk ^ ((row >> 2) & 7) so that the lanes
//                   reading the same k of rows r and r+4 hit distinct banks;
//                   A stored [M,K] stays in this layout (measured faster than
//                   transposing it, by copies or through registers).
template <class TL>
__device__ __forceinline__ int a_swz(int row, int chunk) {
  return chunk ^ ((row >> 2) & TL::SWZ_MASK);
}

// source [R rows][K] (k contiguous) -> row tile of BM rows
template <class TL, bool VEC>
__device__ __forceinline__ void load_rows(uint32_t dst, const float* __restrict__ g, int64_t ld,
                                          int r0, int R, int k0, int K, int tid) {
  constexpr int BM = TL::BM, BK = TL::BK, THREADS = TL::THREADS;
  if constexpr (VEC) {
    constexpr int CPR = BK / 4;  // 16-byte chunks per row
    constexpr int CHUNKS = BM * CPR;
#pragma unroll
    for (int it = 0; it < (CHUNKS + THREADS - 1) / THREADS; ++it) {
      const int q = tid + it * THREADS;
      if (CHUNKS % THREADS != 0 && q >= CHUNKS) break;
      const int row = q / CPR, c = q % CPR;
      const int gr = r0 + row, gk = k0 + c * 4;
      const bool ok = (gr < R) && (gk < K);
      const uint32_t bytes = ok ? (uint32_t)min(4, K - gk) * 4u : 0u;
      const float* src = ok ? g + (int64_t)gr * ld + gk : g;
      cp_async_16(dst + (uint32_t)(row * BK + a_swz<TL>(row, c) * 4) * 4u, src, bytes);
    }
  } else {
    constexpr int ELEMS = BM * BK;
#pragma unroll 4
    for (int it = 0; it < (ELEMS + THREADS - 1) / THREADS; ++it) {
      const int e = tid + it * THREADS;
      if (ELEMS % THREADS != 0 && e >= ELEMS) break;
      const int row = e / BK, kk = e % BK;
      const int gr = r0 + row, gk = k0 + kk;
      const bool ok = (gr < R) && (gk < K);
      const float* src = ok ? g + (int64_t)gr * ld + gk : g;
      const int col = a_swz<TL>(row, kk >> 2) * 4 + (kk & 3);
      cp_async_4(dst + (uint32_t)(row * BK + col) * 4u, src, ok ? 4u : 0u);
    }
  }
}

// source [K][R] (m/n contiguous) -> k-major tile of W columns, row pitch PITCH
template <class TL, bool VEC, int W, int PITCH>
__device__ __forceinline__ void load_kmajor(uint32_t dst, const float* __restrict__ g, int64_t ld,
                                            int r0, int R, int k0, int K, int tid) {
  constexpr int BK = TL::BK, THREADS = TL::THREADS;
  if constexpr (VEC) {
    constexpr int CPR = W / 4;  // 16-byte chunks per k row
    constexpr int CHUNKS = BK * CPR;
#pragma unroll
    for (int it = 0; it < (CHUNKS + THREADS - 1) / THREADS; ++it) {
      const int q = tid + it * THREADS;
      if (CHUNKS % THREADS != 0 && q >= CHUNKS) break;
      const int krow = q / CPR, c = q - krow * CPR;
      const int gk = k0 + krow, gr = r0 + c * 4;
      const bool ok = (gk < K) && (gr < R);
      const uint32_t bytes = ok ? (uint32_t)min(4, R - gr) * 4u : 0u;
      const float* src = ok ? g + (int64_t)gk * ld + gr : g;
      cp_async_16(dst + (uint32_t)(krow * PITCH + c * 4) * 4u, src, bytes);
    }
  } else {
    constexpr int ELEMS = BK * W;
#pragma unroll 4
    for (int it = 0; it < (ELEMS + THREADS - 1) / THREADS; ++it) {
      const int e = tid + it * THREADS;
      if (ELEMS % THREADS != 0 && e >= ELEMS) break;
      const int krow = e / W, rr = e - krow * W;
      const int gk = k0 + krow, gr = r0 + rr;
      const bool ok = (gk < K) && (gr < R);
      const float* src = ok ? g + (int64_t)gk * ld + gr : g;
      cp_async_4(dst + (uint32_t)(krow * PITCH + rr) * 4u, src, ok ? 4u : 0u);
    }
  }
}

// source [R rows][K] (k contiguous) -> k-major tile of W columns, transposed by
// 4-byte copies: lane l reads k = l & 7 of row (l >> 3) of a 4-row group
template <class TL, int W, int PITCH>
__device__ __forceinline__ void load_transpose(uint32_t dst, const float* __restrict__ g,
                                               int64_t ld, int r0, int R, int k0, int K,
                                               int tid) {
  constexpr int BK = TL::BK, THREADS = TL::THREADS;
  const int warp = tid >> 5, lane = tid & 31;
  const int kl = lane & 7, rl = lane >> 3;
  constexpr int GROUPS = (W / 4) * (BK / 8);  // 4-row x 8-k groups
  constexpr int WARPS = THREADS / 32;
#pragma unroll 4
  for (int it = 0; it < (GROUPS + WARPS - 1) / WARPS; ++it) {
    const int grp = warp + it * WARPS;
    if (GROUPS % WARPS != 0 && grp >= GROUPS) break;
    const int rg = grp % (W / 4), kg = grp / (W / 4);
    const int row = rg * 4 + rl, k = kg * 8 + kl;
    const int gr = r0 + row, gk = k0 + k;
    const bool ok = (gr < R) && (gk < K);
    const float* src = ok ? g + (int64_t)gr * ld + gk : g;
    cp_async_4(dst + (uint32_t)(k * PITCH + row) * 4u, src, ok ? 4u : 0u);
  }
}

// ---------------------------------------------------------------- paired FMA
// fma.rn.f32x2: two IEEE fp32 fused multiply-adds (round to nearest even) in
// one instruction on a pair of registers; each half is exactly an fp32 FMA,
// so results keep fp32 semantics.
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t splat2(float x) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ uint64_t pack2(float x, float y) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
  return r;
}
__device__ __forceinline__ float2 unpack2(uint64_t v) {
  float2 f;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(v));
  return f;
}

__device__ __forceinline__ float4 lds128(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}

// Stream-K bookkeeping: the block whose step range contains step x, and the
// first step of block b (G blocks over I steps).
__device__ __forceinline__ int sk_owner(int64_t x, int G, int64_t I) {
  return (int)(((x + 1) * G - 1) / I);
}
__device__ __forceinline__ int64_t sk_start(int b, int G, int64_t I) { return (int64_t)b * I / G; }

// One work item of a block: tile t over K range [kbeg, kend).  seg0 is the
// first step of a stream-K segment; whole marks an item covering all of K.
struct Item {
  int t, kbeg, kend;
  int64_t seg0;
  bool whole;
};

// The persistent walk of block b of G: whole tiles b, b + G, ... below
// dp_tiles, then the block's stream-K step range, one segment per tile it
// touches.
struct Walk {
  int dp_next;
  int64_t sk_it, sk_end, sk_first;
  __device__ __forceinline__ void init(const Params& p, int b, int G) {
    dp_next = b;
    sk_first = sk_it = sk_start(b, G, p.sk_iters);
    sk_end = sk_start(b + 1, G, p.sk_iters);
  }
  template <int BK>
  __device__ __forceinline__ bool next(const Params& p, int G, Item& w) {
    if (dp_next < p.dp_tiles) {
      w.t = dp_next;
      dp_next += G;
      w.kbeg = 0;
      w.kend = p.K;
      w.seg0 = 0;
      w.whole = true;
      return true;
    }
    if (sk_it >= sk_end) return false;
    const int64_t ts = sk_it / p.kiters;
    const int s0 = (int)(sk_it - ts * p.kiters);
    const int64_t left = sk_end - sk_it;
    const int s1 = left < (int64_t)(p.kiters - s0) ? s0 + (int)left : p.kiters;
    w.t = p.dp_tiles + (int)ts;
    w.seg0 = sk_it;
    sk_it += s1 - s0;
    w.kbeg = s0 * BK;
    w.kend = min(p.K, s1 * BK);
    w.whole = s0 == 0 && s1 == p.kiters;
    return true;
  }
};

// Grouped rasterisation of the tile grid (consecutive tiles share B panels
// within a group of group_m tile-rows): the first row and column of tile t.
template <class TL>
__device__ __forceinline__ void tile_origin(const Params& p, int t, int& m0, int& n0) {
  const int per_group = p.group_m * p.tiles_n;
  const int first_m = (t / per_group) * p.group_m;
  const int gsize = min(p.tiles_m - first_m, p.group_m);
  m0 = (first_m + (t % per_group) % gsize) * TL::BM;
  n0 = ((t % per_group) / gsize) * TL::BN;
}

// One k of a lane's 8 x LN block: av holds its 8 A values (rows arow + {0..3},
// arow + 32 + {0..3}); brow points at its B values in the stage's k row
// (columns bcol + 16 h + {0..3}).
template <class TL>
__device__ __forceinline__ void fma_k(uint64_t (&acc)[8][TL::JP], const float (&av)[8],
                                      const float* brow) {
  constexpr int JP = TL::JP, HB = TL::HB;
  uint64_t bp[JP];
#pragma unroll
  for (int h = 0; h < HB; ++h) {
    const ulonglong2 b = *reinterpret_cast<const ulonglong2*>(brow + 16 * h);
    bp[2 * h] = b.x;
    bp[2 * h + 1] = b.y;
  }
  // All eight (a, a) pairs first, then column pair by column pair, the rows
  // alternating between the two 4-row halves: the eight paired FMAs sharing
  // bp[j] follow each other and none waits on the register move that builds
  // its splatted operand.  Measured at 4096^3 against row by row (i outer, j
  // inner): +5 %; rows in order 0..7: -0.1 %; other interleavings: -0.5 to
  // -2.6 %.
  uint64_t ap[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) ap[i] = splat2(av[i]);
  constexpr int ORD[8] = {0, 4, 1, 5, 2, 6, 3, 7};
#pragma unroll
  for (int j = 0; j < JP; ++j)
#pragma unroll
    for (int ii = 0; ii < 8; ++ii) acc[ORD[ii]][j] = ffma2(ap[ORD[ii]], bp[j], acc[ORD[ii]][j]);
}

// Barrier over the threads that compute (N = 0: the whole block; else the
// first N threads, named barrier 1, the other warps not taking part).
template <int N>
__device__ __forceinline__ void compute_sync() {
  if constexpr (N == 0) __syncthreads();
  else asm volatile("bar.sync 1, %0;" ::"n"(N) : "memory");
}

// Output row (within the tile) of a lane's i-th row: blocks of four, rows
// arow + {0..3} and arow + 32 + {0..3} (RI false), or interleaved by eight,
// rows arow + 8 i (RI true, the layout that reads a 128-byte-swizzled row
// tile without bank conflicts).
template <bool RI>
__device__ __forceinline__ int lane_row(int arow, int i) {
  return RI ? arow + 8 * i : arow + (i < 4 ? i : 32 + i - 4);
}

// The end of a work item.  A tile shared between blocks (not `whole`, a
// persistent launch) has its partial sums published; only its last
// contributor goes on, with the sum of all contributions.  Then the epilogue
// (alpha, beta, bias, activation) stores the lane's block of C, or, in a
// split launch, its raw sums in slice blockIdx.z of `partial`.  SYNC: the
// barrier over the computing threads (compute_sync); RI: lane_row's layout.
template <class TL, int KIND, int SYNC, bool RI = false>
__device__ __forceinline__ void finish_item(const Params& p, uint64_t (&acc)[8][TL::JP],
                                            const Item& w, int64_t sk_first, int m0, int n0,
                                            float* Cg, int tid, int arow, int bcol, int& s_last) {
  constexpr int BM = TL::BM, BN = TL::BN, THREADS = TL::THREADS, JP = TL::JP, HB = TL::HB;
  if constexpr (KIND == KIND_PERSIST) {
    if (!w.whole) {
      // Every contributor stores its partial sums (warp-coalesced: float4 j
      // of thread tid at [j][tid]) in its slot -- 0 for the segment a block
      // starts with, 1 for the one it ends with -- then counts itself in.
      // The last to arrive adds all segments in K order (so the result does
      // not depend on arrival order) and stores the tile.
      const int G = gridDim.x;
      const int slot = w.seg0 == sk_first ? 0 : 1;
      float4* mine = reinterpret_cast<float4*>(p.sk_ws) +
                     (int64_t)(blockIdx.x * 2 + slot) * (BM * BN / 4);
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int h = 0; h < HB; ++h) {
          const float2 lo = unpack2(acc[i][2 * h]), hi = unpack2(acc[i][2 * h + 1]);
          mine[(i * HB + h) * THREADS + tid] = make_float4(lo.x, lo.y, hi.x, hi.y);
        }
      __threadfence();
      compute_sync<SYNC>();
      const int64_t x0 = (int64_t)(w.t - p.dp_tiles) * p.kiters;
      const int c_lo = sk_owner(x0, G, p.sk_iters);
      const int c_hi = sk_owner(x0 + p.kiters - 1, G, p.sk_iters);
      if (tid == 0) {
        const unsigned int before = atomicAdd(p.sk_cnt + (w.t - p.dp_tiles), 1u);
        s_last = before == (unsigned int)(c_hi - c_lo);
      }
      compute_sync<SYNC>();
      const bool last = s_last != 0;
      // (tid 0 writes s_last again only past the first barrier of the next
      // shared tile, which every computing thread reaches after this read)
      if (!last) return;
      __threadfence();
      float sum[8][JP][2];
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < JP; ++j) sum[i][j][0] = sum[i][j][1] = 0.f;
      for (int c = c_lo; c <= c_hi; ++c) {
        const int cs = sk_start(c, G, p.sk_iters) >= x0 ? 0 : 1;
        const float4* part = reinterpret_cast<const float4*>(p.sk_ws) +
                             (int64_t)(c * 2 + cs) * (BM * BN / 4);
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int h = 0; h < HB; ++h) {
            const float4 v = __ldcg(part + (i * HB + h) * THREADS + tid);
            sum[i][2 * h][0] += v.x; sum[i][2 * h][1] += v.y;
            sum[i][2 * h + 1][0] += v.z; sum[i][2 * h + 1][1] += v.w;
          }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < JP; ++j) acc[i][j] = pack2(sum[i][j][0], sum[i][j][1]);
    }
  }

  // epilogue: lane columns bcol + 16 h + {0..3} (pairs 2h, 2h + 1)
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int gm = m0 + lane_row<RI>(arow, i);
    if (gm >= p.M) continue;
#pragma unroll
    for (int h = 0; h < HB; ++h) {
      const int gn = n0 + bcol + h * 16;
      const float2 lo = unpack2(acc[i][2 * h]), hi = unpack2(acc[i][2 * h + 1]);
      const float v[4] = {lo.x, lo.y, hi.x, hi.y};
      if constexpr (KIND == KIND_SPLIT) {
        float* dst = p.partial + ((int64_t)blockIdx.z * p.M + gm) * p.N + gn;
        if (gn + 3 < p.N && (p.N & 3) == 0) {
          *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (gn + j < p.N) dst[j] = v[j];
        }
      } else {
        float* dst = Cg + (int64_t)gm * p.ldc + gn;
        const bool vec_ok = p.c_vec && (gn + 3 < p.N);
        const bool epi = p.ep.bias != nullptr || p.ep.act != 0;
        if (vec_ok) {
          float4 o;
          if (p.beta != 0.f) {
            const float4 c = *reinterpret_cast<const float4*>(dst);
            o = make_float4(__fmaf_rn(p.alpha, v[0], p.beta * c.x),
                            __fmaf_rn(p.alpha, v[1], p.beta * c.y),
                            __fmaf_rn(p.alpha, v[2], p.beta * c.z),
                            __fmaf_rn(p.alpha, v[3], p.beta * c.w));
          } else {
            o = make_float4(p.alpha * v[0], p.alpha * v[1], p.alpha * v[2], p.alpha * v[3]);
          }
          if (epi) {
            o.x = apply_epilogue<float>(o.x, p.ep, gn);
            o.y = apply_epilogue<float>(o.y, p.ep, gn + 1);
            o.z = apply_epilogue<float>(o.z, p.ep, gn + 2);
            o.w = apply_epilogue<float>(o.w, p.ep, gn + 3);
          }
          *reinterpret_cast<float4*>(dst) = o;
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (gn + j < p.N) {
              float o = (p.beta != 0.f) ? __fmaf_rn(p.alpha, v[j], p.beta * dst[j])
                                        : p.alpha * v[j];
              if (epi) o = apply_epilogue<float>(o, p.ep, gn + j);
              dst[j] = o;
            }
          }
        }
      }
    }
  }
}

template <class TL, bool A_K, bool B_K, bool VEC, int KIND>
__global__ void __launch_bounds__(TL::THREADS, TL::MIN_BLOCKS) sgemm_ffma_kernel(const Params p) {
  constexpr int BM = TL::BM, BK = TL::BK;
  constexpr int WARPS_N = TL::WARPS_N, APAD = TL::APAD, BPAD = TL::BPAD;
  constexpr int A_FLOATS = TL::A_FLOATS, STAGE_FLOATS = TL::STAGE_FLOATS;
  constexpr int JP = TL::JP, NST = TL::NSTAGES;
  // (the previous kernel in the stream completes before any global access)
  pdl_wait();
  pdl_trigger();
  extern __shared__ __align__(16) float smem[];
  __shared__ int s_last;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int wm = (warp / WARPS_N) * 64;          // warp's first row in the tile
  const int wn = (warp % WARPS_N) * TL::WARP_N;  // warp's first column
  const int ty = lane >> 2, tx = lane & 3;
  const int arow = wm + ty * 4;     // lane rows: arow + {0..3}, arow + 32 + {0..3}
  const int bcol = wn + tx * 4;     // lane cols: bcol + 16 h + {0..3}, h < HB
  const int aswz = (arow >> 2) & TL::SWZ_MASK;  // row-tile chunk permutation, same for all 8 lane rows

  const float* const Ag = p.A + (int64_t)blockIdx.y * p.stride_a;
  const float* const Bg = p.B + (int64_t)blockIdx.y * p.stride_b;
  float* const Cg = p.C + (int64_t)blockIdx.y * p.stride_c;
  const uint32_t sbase = smem_u32(smem);

  // work state: non-persistent blocks do one item; persistent blocks walk
  // their whole tiles, then their stream-K step range
  const int G = gridDim.x;
  Walk walk = {};
  if constexpr (KIND == KIND_PERSIST) walk.init(p, blockIdx.x, G);
  bool first_item = true;

  // acc[i][jp] holds the outputs (row i, lane columns 2jp and 2jp+1) as a pair
  uint64_t acc[8][JP];

  for (;;) {
    Item w;
    if constexpr (KIND != KIND_PERSIST) {
      if (!first_item) break;
      w.t = blockIdx.x;
      w.kbeg = blockIdx.z * p.k_slice;
      w.kend = min(p.K, w.kbeg + p.k_slice);
      w.seg0 = 0;
      w.whole = true;
    } else {
      if (!walk.next<BK>(p, G, w)) break;
    }
    first_item = false;
    int m0, n0;
    tile_origin<TL>(p, w.t, m0, n0);
    const int kbeg = w.kbeg, kend = w.kend;
    const int nk = (kend - kbeg + BK - 1) / BK;

    auto stage_load = [&](int s, int k0) {
      const uint32_t st = sbase + (uint32_t)(s * STAGE_FLOATS) * 4u;
      if constexpr (A_K) load_rows<TL, VEC>(st, Ag, p.lda, m0, p.M, k0, kend, tid);
      else load_kmajor<TL, VEC, BM, APAD>(st, Ag, p.lda, m0, p.M, k0, kend, tid);
      const uint32_t sb = st + A_FLOATS * 4u;
      if constexpr (B_K) load_transpose<TL, TL::BN, BPAD>(sb, Bg, p.ldb, n0, p.N, k0, kend, tid);
      else load_kmajor<TL, VEC, TL::BN, BPAD>(sb, Bg, p.ldb, n0, p.N, k0, kend, tid);
    };

#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < JP; ++j) acc[i][j] = 0ull;

    if constexpr (KIND == KIND_PERSIST) __syncthreads();  // the previous item's stages are free
#pragma unroll
    for (int s = 0; s < NST - 1; ++s) {
      if (s < nk) stage_load(s, kbeg + s * BK);
      cp_async_commit();
    }

    for (int kt = 0; kt < nk; ++kt) {
      cp_async_wait<NST - 2>();
      __syncthreads();  // stage kt visible to all; stage kt-1 fully consumed
      {
        const int nxt = kt + NST - 1;
        if (nxt < nk) stage_load(nxt % NST, kbeg + nxt * BK);
        cp_async_commit();
      }
      const float* As = smem + (kt % NST) * STAGE_FLOATS;
      const float* Bs = As + A_FLOATS;
#pragma unroll KC_UNROLL
      for (int kc = 0; kc < BK / 4; ++kc) {
        float a[8][4];  // a[i][kk]: row i, k = 4kc + kk (row-tile A)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int k = kc * 4 + kk;
          float av[8];
          if constexpr (A_K) {
            // two k at a time (64-bit loads) keeps 16 rather than 32 A values live
            if ((kk & 1) == 0) {
              const float* base = As + arow * BK + ((kc ^ aswz) * 4) + kk;
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float2 v =
                    *reinterpret_cast<const float2*>(base + (i < 4 ? i : 32 + i - 4) * BK);
                a[i][kk] = v.x; a[i][kk + 1] = v.y;
              }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) av[i] = a[i][kk];
          } else {
            const float4 lo = lds128(As + k * APAD + arow);
            const float4 hi = lds128(As + k * APAD + arow + 32);
            av[0] = lo.x; av[1] = lo.y; av[2] = lo.z; av[3] = lo.w;
            av[4] = hi.x; av[5] = hi.y; av[6] = hi.z; av[7] = hi.w;
          }
          fma_k<TL>(acc, av, Bs + k * BPAD + bcol);
        }
      }
    }
    cp_async_wait<0>();

    finish_item<TL, KIND, 0>(p, acc, w, walk.sk_first, m0, n0, Cg, tid, arow, bcol, s_last);
  }
}

// ---------------------------------------------------------------- warp-specialised
// Variant for a B stored k-major ([K, N]) and an A stored either way, all rows
// 16-byte aligned (the layouts the packing pre-pass writes, and the narrow
// tile's A as given).  One extra warp streams both operand tiles of every K
// step into the NST-stage ring by TMA, each stage's arrival counted on its
// `full` mbarrier; the computing warps wait only for the stage they need and
// release it with one arrival per warp on its `empty` mbarrier.  No
// block-wide barrier and no copy instruction sits in the main loop, and in a
// persistent launch the loads of the next item's first stages overlap the
// current item's epilogue.  Tile parts past M, N or K read as zeros (the
// tensor maps' out-of-range fill).
//
// A stored [K, M] (A_K false) arrives as BK dense rows of BM floats.  A
// stored [M, K] (A_K true, K step 32) arrives as BM rows of 32 floats = 128
// bytes with the tensor unit's 128-byte swizzle (16-byte chunk j of row r at
// chunk j ^ (r & 7)); a lane then owns rows interleaved by eight (lane_row),
// so that the eight row groups of a warp read eight different chunks: no bank
// conflicts.
//
// KIND_PERSIST walks whole tiles and then a stream-K step range (Walk);
// KIND_SPLIT and KIND_TILE give every block one item (tile blockIdx.x, K
// slice blockIdx.z).  Every wait is bounded: a warp whose wait expires stops
// computing (the status word then holds GEMM_ERR_TIMEOUT) but still walks its
// items, so the computing warps' barriers stay matched; the producer drains
// its copies in flight.
template <class TL>
struct WsCfg {
  static constexpr int A_BYTES = TL::BM * TL::BK * 4;  // [BK][BM] or [BM][BK]
  static constexpr int B_BYTES = TL::BN * TL::BK * 4;  // [BK][BN]
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int THREADS = TL::THREADS + 32;
  static constexpr int SMEM_BYTES = TL::NSTAGES * STAGE_BYTES + 1024;  // + alignment slack
  static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "stage alignment");
};

template <class TL, bool A_K, int KIND>
__global__ void __launch_bounds__(TL::THREADS + 32, TL::MIN_BLOCKS)
    sgemm_ws_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB, const Params p) {
  constexpr int BM = TL::BM, BN = TL::BN, BK = TL::BK, NST = TL::NSTAGES, JP = TL::JP;
  constexpr int WARPS = TL::THREADS / 32;
  static_assert(!A_K || BK == 32, "row tiles of A: 128-byte rows");
  using WC = WsCfg<TL>;
  extern __shared__ __align__(1024) uint8_t ws_smem[];
  __shared__ __align__(8) uint64_t bars[2 * NST];
  __shared__ uint32_t s_abort;
  __shared__ int s_last;
  const uint32_t raw = smem_u32(ws_smem);
  const uint32_t ring = (raw + 1023u) & ~1023u;
  const float* const ring_f = reinterpret_cast<const float*>(ws_smem + (ring - raw));
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * (uint32_t)s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (uint32_t)(NST + s); };
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), WARPS);
    }
    s_abort = 0u;
    fence_mbar_init();
  }
  __syncthreads();
  // (the previous kernel in the stream completes before any global access)
  pdl_wait();
  pdl_trigger();
  const WaitCtl wc{p.status, &s_abort, p.timeout_ns};
  const int G = gridDim.x;
  Walk walk = {};
  if constexpr (KIND == KIND_PERSIST) walk.init(p, blockIdx.x, G);
  bool single_done = false;
  // the next work item of this block (the same sequence for every warp)
  auto next = [&](Item& w) -> bool {
    if constexpr (KIND == KIND_PERSIST) {
      return walk.next<BK>(p, G, w);
    } else {
      if (single_done) return false;
      single_done = true;
      w.t = blockIdx.x;
      w.kbeg = blockIdx.z * p.k_slice;
      w.kend = min(p.K, w.kbeg + p.k_slice);
      w.seg0 = 0;
      w.whole = true;
      return w.kbeg < w.kend;
    }
  };
  Item w;

  if (warp == WARPS) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      int stage = 0;
      uint32_t phase = 0, pending = 0, pend_phase = 0;  // per stage: last load issued / its parity
      bool ok = true, first = true;
      while (ok && next(w)) {
        int m0, n0;
        tile_origin<TL>(p, w.t, m0, n0);
        for (int k0 = w.kbeg; k0 < w.kend; k0 += BK) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, wc)) { ok = false; break; }
          // (test hook: the first stage's loads are never issued)
          const bool skip = first && p.fault_injection == 1;
          first = false;
          if (!skip) {
            const uint32_t sa = ring + (uint32_t)(stage * WC::STAGE_BYTES);
            mbar_arrive_expect_tx(full_bar(stage), WC::STAGE_BYTES);
            if constexpr (A_K) tma_load_3d(sa, &tmA, k0, m0, 0, full_bar(stage));
            else tma_load_3d(sa, &tmA, m0, k0, 0, full_bar(stage));
            tma_load_3d(sa + WC::A_BYTES, &tmB, n0, k0, 0, full_bar(stage));
            pending |= 1u << stage;
            pend_phase = (pend_phase & ~(1u << stage)) | (phase << stage);
          }
          if (++stage == NST) { stage = 0; phase ^= 1u; }
        }
      }
      // every load issued lands before the block's shared memory is released
      for (int s = 0; s < NST; ++s)
        if (pending & (1u << s)) mbar_wait_drain(full_bar(s), (pend_phase >> s) & 1u, p.timeout_ns);
    }
    return;
  }

  // -------------------------------------------------------------- computing warps
  const int wm = (warp / TL::WARPS_N) * 64;          // warp's first row in the tile
  const int wn = (warp % TL::WARPS_N) * TL::WARP_N;  // warp's first column
  const int ty = lane >> 2, tx = lane & 3;
  // lane rows: lane_row<A_K>(arow, i), i < 8; lane cols: bcol + 16 h + {0..3}
  const int arow = A_K ? wm + ty : wm + ty * 4;
  const int bcol = wn + tx * 4;
  uint64_t acc[8][JP];
  int stage = 0;
  uint32_t phase = 0;
  bool failed = false;
  while (next(w)) {
    int m0, n0;
    tile_origin<TL>(p, w.t, m0, n0);
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < JP; ++j) acc[i][j] = 0ull;
    for (int k0 = w.kbeg; k0 < w.kend; k0 += BK) {
      if (!failed) failed = !__all_sync(0xffffffffu, mbar_wait(full_bar(stage), phase, wc));
      if (!failed) {
        const float* As = ring_f + stage * (WC::STAGE_BYTES / 4);
        const float* Bs = As + BM * BK;
        if constexpr (A_K) {
          // row r = arow + 8 i holds its k = 4 c + e at chunk c ^ (r & 7) = c ^ ty:
          // one 128-bit load a row gives four k
          const float* Ar = As + arow * BK;
#pragma unroll
          for (int kc = 0; kc < BK / 4; ++kc) {
            const int ch = ((kc ^ ty) & 7) * 4;
            float4 v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = lds128(Ar + i * 8 * BK + ch);
            const float a0[8] = {v[0].x, v[1].x, v[2].x, v[3].x, v[4].x, v[5].x, v[6].x, v[7].x};
            const float a1[8] = {v[0].y, v[1].y, v[2].y, v[3].y, v[4].y, v[5].y, v[6].y, v[7].y};
            const float a2[8] = {v[0].z, v[1].z, v[2].z, v[3].z, v[4].z, v[5].z, v[6].z, v[7].z};
            const float a3[8] = {v[0].w, v[1].w, v[2].w, v[3].w, v[4].w, v[5].w, v[6].w, v[7].w};
            fma_k<TL>(acc, a0, Bs + (kc * 4 + 0) * BN + bcol);
            fma_k<TL>(acc, a1, Bs + (kc * 4 + 1) * BN + bcol);
            fma_k<TL>(acc, a2, Bs + (kc * 4 + 2) * BN + bcol);
            fma_k<TL>(acc, a3, Bs + (kc * 4 + 3) * BN + bcol);
          }
        } else {
#pragma unroll KC_UNROLL
          for (int kc = 0; kc < BK / 4; ++kc) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const int k = kc * 4 + kk;
              const float4 lo = lds128(As + k * BM + arow);
              const float4 hi = lds128(As + k * BM + arow + 32);
              const float av[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
              fma_k<TL>(acc, av, Bs + k * BN + bcol);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_bar(stage));
      }
      if (++stage == NST) { stage = 0; phase ^= 1u; }
    }
    finish_item<TL, KIND, TL::THREADS, A_K>(p, acc, w, walk.sk_first, m0, n0, p.C, tid, arow,
                                            bcol, s_last);
  }
}

// The warp-specialised launch of `grid` blocks of kind KIND.
template <class TL, bool A_K, int KIND>
cudaError_t launch_ws(const Params& p, const SgemmArgs& a, dim3 grid, cudaStream_t stream) {
  using WC = WsCfg<TL>;
  // A as [K, M] (boxes of BK rows x BM) or [M, K] (BM rows x 32, swizzled),
  // B as [K, N] (BK rows x BN), fp32
  CUtensorMap mA, mB;
  const bool okA =
      A_K ? make_map(&mA, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.A, a.M, a.K, a.lda, TL::BK, TL::BM,
                     CU_TENSOR_MAP_SWIZZLE_128B, 1, 0, 4)
          : make_map(&mA, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.A, a.K, a.M, a.lda, TL::BM, TL::BK,
                     CU_TENSOR_MAP_SWIZZLE_NONE, 1, 0, 4);
  if (!okA || !make_map(&mB, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.B, a.K, a.N, a.ldb, TL::BN,
                        TL::BK, CU_TENSOR_MAP_SWIZZLE_NONE, 1, 0, 4))
    return cudaErrorNotSupported;
  auto kern = sgemm_ws_kernel<TL, A_K, KIND>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       WC::SMEM_BYTES);
  if (e == cudaSuccess && TL::MIN_BLOCKS > 1)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, grid, dim3(WC::THREADS), WC::SMEM_BYTES, stream, 1, mA, mB, p);
}

template <class TL, bool A_K, bool B_K, bool VEC, int KIND>
cudaError_t launch_one(const Params& p, dim3 grid, cudaStream_t stream) {
  auto kern = sgemm_ffma_kernel<TL, A_K, B_K, VEC, KIND>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       TL::SMEM_BYTES);
  // several resident blocks need the largest shared-memory carve-out
  if (e == cudaSuccess && TL::MIN_BLOCKS > 1)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, grid, dim3(TL::THREADS), TL::SMEM_BYTES, stream, 1, p);
}

// (PERSIST: the stream-K launch, instantiated only for tiles that use it)
template <class TL, bool A_K, bool B_K, bool PERSIST>
cudaError_t launch_vs(const Params& p, bool vec, int kind, dim3 grid, cudaStream_t s) {
  if (kind == KIND_PERSIST) {
    if constexpr (PERSIST) {
      return vec ? launch_one<TL, A_K, B_K, true, KIND_PERSIST>(p, grid, s)
                 : launch_one<TL, A_K, B_K, false, KIND_PERSIST>(p, grid, s);
    } else {
      return cudaErrorInvalidValue;
    }
  }
  if (vec) {
    if (kind == KIND_SPLIT) return launch_one<TL, A_K, B_K, true, KIND_SPLIT>(p, grid, s);
    return launch_one<TL, A_K, B_K, true, KIND_TILE>(p, grid, s);
  }
  if (kind == KIND_SPLIT) return launch_one<TL, A_K, B_K, false, KIND_SPLIT>(p, grid, s);
  return launch_one<TL, A_K, B_K, false, KIND_TILE>(p, grid, s);
}

// The whole launch for tile TL (host side of launch_sgemm).
template <class TL, bool PERSIST>
cudaError_t launch_sgemm_t(const SgemmArgs& a, LaunchCtx& ctx) {
  constexpr int BM = TL::BM, BN = TL::BN, BK = TL::BK;
  Params p;
  p.A = a.A; p.B = a.B; p.C = a.C; p.partial = a.partial;
  p.lda = a.lda; p.ldb = a.ldb; p.ldc = a.ldc;
  p.M = a.M; p.N = a.N; p.K = a.K;
  p.k_slice = a.splits > 1 ? a.k_slice : a.K;
  p.tiles_m = (a.M + BM - 1) / BM;
  p.tiles_n = (a.N + BN - 1) / BN;
  {
    const int64_t panel = (int64_t)BM * (a.splits > 1 ? a.k_slice : a.K) * 4;
    int64_t g = panel > 0 ? RASTER_L2_BYTES / panel : p.tiles_m;
    if (g < 1) g = 1;
    if (g > p.tiles_m) g = p.tiles_m;
    p.group_m = (int)g;
  }
  p.alpha = a.alpha; p.beta = a.beta;
  p.ep = a.ep;
  p.status = ctx.status;
  p.timeout_ns = ctx.timeout_ns;
  p.fault_injection = a.fault_injection;
  const int batch = a.batch > 1 ? a.batch : 1;
  if (batch > 1 && (a.splits > 1 || batch > 65535)) return cudaErrorInvalidValue;
  p.stride_a = batch > 1 ? a.stride_a : 0;
  p.stride_b = batch > 1 ? a.stride_b : 0;
  p.stride_c = batch > 1 ? a.stride_c : 0;
  // 16-byte staging needs 16-byte aligned rows in both operands and every
  // batch entry; the epilogue's float4 accesses need the same of C.
  const bool vec = ((reinterpret_cast<uintptr_t>(a.A) | reinterpret_cast<uintptr_t>(a.B)) &
                    15u) == 0 &&
                   (a.lda % 4) == 0 && (a.ldb % 4) == 0 && (p.stride_a % 4) == 0 &&
                   (p.stride_b % 4) == 0;
  p.c_vec = (reinterpret_cast<uintptr_t>(a.C) & 15u) == 0 && (a.ldc % 4) == 0 &&
            (p.stride_c % 4) == 0;
  const bool split = a.splits > 1;
  const int tiles = p.tiles_m * p.tiles_n;
  int kind = split ? KIND_SPLIT : KIND_TILE;
  dim3 grid(tiles, batch, split ? a.splits : 1);
  p.dp_tiles = 0; p.kiters = 0; p.sk_iters = 0; p.sk_ws = nullptr; p.sk_cnt = nullptr;
  if (a.sk_blocks > 0) {
    // persistent: all but the last one to two rounds of whole tiles go to
    // blocks in turn; the rest (every tile, with fewer tiles than blocks) are
    // shared out by K steps, each block's range non-empty
    const int G = a.sk_blocks;
    p.kiters = (a.K + BK - 1) / BK;
    if (split || batch > 1 || (int64_t)tiles * p.kiters < G || !a.sk_ws || !a.sk_cnt)
      return cudaErrorInvalidValue;
    kind = KIND_PERSIST;
    p.dp_tiles = tiles >= 2 * G ? (tiles / G - 1) * G : 0;
    p.sk_iters = (int64_t)(tiles - p.dp_tiles) * p.kiters;
    p.sk_ws = a.sk_ws;
    p.sk_cnt = a.sk_cnt;
    grid = dim3(G, 1, 1);
  }
  const bool A_K = !a.transA, B_K = a.transB;
  cudaError_t e = cudaErrorInvalidValue;
  // Warp-specialised TMA staging, for tiles with 8 x 8 lane blocks (with the
  // extra warp ptxas holds a thread to 168 registers, where the 8 x 16 block
  // spills), one GEMM, aligned rows, B stored [K, N]:
  //  - tiles with a persistent launch (128 x 128, 128 x 64): A stored [K, M]
  //    (packed so on large problems); persistent over the stream-K plan, one
  //    block per tile without one, or one per (tile, K slice);
  //  - the narrow tile (256 x 32, K step 32): A stored either way, one block
  //    per tile or per (tile, K slice).
  constexpr bool WS_P = PERSIST && TL::LN == 8;
  constexpr bool WS_N = !PERSIST && TL::LN == 8 && TL::BK == 32;
  const bool ws_ok = a.ws && batch == 1 && vec && !B_K;
  if (WS_P && ws_ok && !A_K) {
    if (split) {
      if constexpr (WS_P) e = launch_ws<TL, false, KIND_SPLIT>(p, a, grid, ctx.stream);
    } else {
      if (kind != KIND_PERSIST) {
        p.kiters = (a.K + BK - 1) / BK;
        p.dp_tiles = tiles;
        grid = dim3(tiles, 1, 1);
      }
      if constexpr (WS_P) e = launch_ws<TL, false, KIND_PERSIST>(p, a, grid, ctx.stream);
    }
  } else if (WS_N && ws_ok) {
    if constexpr (WS_N) {
      if (A_K)
        e = split ? launch_ws<TL, true, KIND_SPLIT>(p, a, grid, ctx.stream)
                  : launch_ws<TL, true, KIND_TILE>(p, a, grid, ctx.stream);
      else
        e = split ? launch_ws<TL, false, KIND_SPLIT>(p, a, grid, ctx.stream)
                  : launch_ws<TL, false, KIND_TILE>(p, a, grid, ctx.stream);
    }
  } else if (A_K && !B_K) e = launch_vs<TL, true, false, PERSIST>(p, vec, kind, grid, ctx.stream);
  else if (!A_K && !B_K) e = launch_vs<TL, false, false, PERSIST>(p, vec, kind, grid, ctx.stream);
  else if (A_K && B_K) e = launch_vs<TL, true, true, PERSIST>(p, vec, kind, grid, ctx.stream);
  else e = launch_vs<TL, false, true, PERSIST>(p, vec, kind, grid, ctx.stream);
  ctx.grid = (int)(grid.x * grid.y * grid.z);
  if (e == cudaSuccess) ctx.launches++;
  return e;
}

}  // namespace
}  // namespace gb300
