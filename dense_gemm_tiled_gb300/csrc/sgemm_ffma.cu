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
// Tile: 128 x 128 outputs per block, K step 32, 256 threads (8 warps as 2 x 4,
// each warp 64 x 32, each lane 8 x 8 outputs split into 4-wide groups), two
// blocks per SM.  The inner product runs on Blackwell's paired FP32 FMA
// (fma.rn.f32x2): one instruction updates two adjacent outputs of a lane, which
// halves the issue slots the FMAs take -- the original kernel was bound by
// instruction issue, not by the FP32 lanes.  Each pair lane is an IEEE fp32 FMA
// (round to nearest even); no fast-math, denormals kept.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace gb300 {
namespace {

constexpr int BM = SG_BM, BN = SG_BN, BK = SG_BK;
constexpr int STAGES = 3;
constexpr int THREADS = 256;
constexpr int PAD = BN + 4;                 // k-major tile rows padded: conflict-free transposing writes
constexpr int TILE_FLOATS = BK * PAD;       // 16.5 KiB per operand per stage
constexpr int STAGE_FLOATS = 2 * TILE_FLOATS;
constexpr int SMEM_BYTES = STAGES * STAGE_FLOATS * 4;  // 99 KiB: two blocks per SM
constexpr int GROUP_M = 8;  // tile rasterisation: 8 tile-rows walked together
static_assert(BM == BN, "square block tile");

// Compile-time tuning knobs.
//  GB300_SG_MIN_BLOCKS  blocks per SM the register budget is sized for
//  GB300_SG_KC_UNROLL   unrolling of the 4-k chunk loop
//  GB300_SG_A_T         1: an A stored [M,K] is transposed into a k-major tile on
//                       the way in (as B stored [N,K] always is)
//  GB300_SG_MATH        0: scalar FMA; 1: paired FMA, A value splatted into both
//                       halves; 2: paired FMA on (row, row+1) x (col, col+1)
//                       pairs plus the column-swapped pair (no splat; needs a
//                       k-major A tile)
#ifndef GB300_SG_MIN_BLOCKS
#define GB300_SG_MIN_BLOCKS 1
#endif
#ifndef GB300_SG_KC_UNROLL
#define GB300_SG_KC_UNROLL 8
#endif
#ifndef GB300_SG_A_T
#define GB300_SG_A_T 0
#endif
#ifndef GB300_SG_MATH
#define GB300_SG_MATH 1
#endif
constexpr int KC_UNROLL = GB300_SG_KC_UNROLL;
constexpr bool A_TRANSPOSE = GB300_SG_A_T != 0;
constexpr int MATH = GB300_SG_MATH;

struct Params {
  const float* A;
  const float* B;
  float* C;
  float* partial;
  int64_t lda, ldb, ldc;
  int M, N, K;
  int k_slice;
  int tiles_m, tiles_n;
  float alpha, beta;
};

// ---------------------------------------------------------------- staging
// Two tile layouts per operand and stage:
//  "k-major" tile : 32 rows (k) x 128 (m or n), rows padded to 132 floats; an
//                   operand stored with m/n contiguous (A[K,M], B[K,N]) is copied
//                   row by row with 16-byte copies; one stored with k contiguous
//                   (A[M,K], B[N,K]) can be transposed into it on the way in with
//                   4-byte copies -- the transposing write of "Metal GEMM Kernels
//                   for LoRA Training", section 3, done by the async-copy unit.
//                   A warp then reads 4 rows x 32 bytes of global memory and,
//                   thanks to the padding, writes 32 distinct banks.
//  "row" tile     : 128 rows (m) x 32 k, 128-byte rows whose eight 16-byte chunks
//                   are permuted by chunk ^ ((row >> 2) & 7) so that the lanes
//                   reading the same k of rows r and r+4 hit distinct banks;
//                   filled from A[M,K] with 16-byte copies.
__device__ __forceinline__ int a_swz(int row, int chunk) { return chunk ^ ((row >> 2) & 7); }

// source [R rows][K] (k contiguous) -> row tile
template <bool VEC>
__device__ __forceinline__ void load_rows(uint32_t dst, const float* __restrict__ g, int64_t ld,
                                          int r0, int R, int k0, int K, int tid) {
  if constexpr (VEC) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int q = tid + r * THREADS;
      const int row = q >> 3, c = q & 7;
      const int gr = r0 + row, gk = k0 + c * 4;
      const bool ok = (gr < R) && (gk < K);
      const uint32_t bytes = ok ? (uint32_t)min(4, K - gk) * 4u : 0u;
      const float* src = ok ? g + (int64_t)gr * ld + gk : g;
      cp_async_16(dst + (uint32_t)(row * BK + a_swz(row, c) * 4) * 4u, src, bytes);
    }
  } else {
#pragma unroll 4
    for (int r = 0; r < 16; ++r) {
      const int e = tid + r * THREADS;
      const int row = e >> 5, kk = e & 31;
      const int gr = r0 + row, gk = k0 + kk;
      const bool ok = (gr < R) && (gk < K);
      const float* src = ok ? g + (int64_t)gr * ld + gk : g;
      const int col = a_swz(row, kk >> 2) * 4 + (kk & 3);
      cp_async_4(dst + (uint32_t)(row * BK + col) * 4u, src, ok ? 4u : 0u);
    }
  }
}

// source [K][R] (m/n contiguous) -> k-major tile
template <bool VEC>
__device__ __forceinline__ void load_kmajor(uint32_t dst, const float* __restrict__ g, int64_t ld,
                                            int r0, int R, int k0, int K, int tid) {
  if constexpr (VEC) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int q = tid + r * THREADS;
      const int krow = q >> 5, c = q & 31;
      const int gk = k0 + krow, gr = r0 + c * 4;
      const bool ok = (gk < K) && (gr < R);
      const uint32_t bytes = ok ? (uint32_t)min(4, R - gr) * 4u : 0u;
      const float* src = ok ? g + (int64_t)gk * ld + gr : g;
      cp_async_16(dst + (uint32_t)(krow * PAD + c * 4) * 4u, src, bytes);
    }
  } else {
#pragma unroll 4
    for (int r = 0; r < 16; ++r) {
      const int e = tid + r * THREADS;
      const int krow = e >> 7, rr = e & 127;
      const int gk = k0 + krow, gr = r0 + rr;
      const bool ok = (gk < K) && (gr < R);
      const float* src = ok ? g + (int64_t)gk * ld + gr : g;
      cp_async_4(dst + (uint32_t)(krow * PAD + rr) * 4u, src, ok ? 4u : 0u);
    }
  }
}

// source [R rows][K] (k contiguous) -> k-major tile, transposed by 4-byte copies:
// lane l reads k = l & 7 of row (l >> 3) of a 4-row group
__device__ __forceinline__ void load_transpose(uint32_t dst, const float* __restrict__ g,
                                               int64_t ld, int r0, int R, int k0, int K,
                                               int tid) {
  const int warp = tid >> 5, lane = tid & 31;
  const int kl = lane & 7, rl = lane >> 3;
#pragma unroll 4
  for (int r = 0; r < 16; ++r) {
    const int grp = r * 8 + warp;  // 0..127: 32 row-groups of 4 x 4 k-groups of 8
    const int row = (grp & 31) * 4 + rl, k = (grp >> 5) * 8 + kl;
    const int gr = r0 + row, gk = k0 + k;
    const bool ok = (gr < R) && (gk < K);
    const float* src = ok ? g + (int64_t)gr * ld + gk : g;
    cp_async_4(dst + (uint32_t)(k * PAD + row) * 4u, src, ok ? 4u : 0u);
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
__device__ __forceinline__ uint64_t swap2(uint64_t v) {
  uint64_t r;
  asm("{\n\t.reg .b32 lo, hi;\n\tmov.b64 {lo, hi}, %1;\n\tmov.b64 %0, {hi, lo};\n\t}"
      : "=l"(r) : "l"(v));
  return r;
}
__device__ __forceinline__ float2 unpack2(uint64_t v) {
  float2 f;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(v));
  return f;
}
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ float4 lds128(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}

// Accumulators of one lane's 8 x 8 block, in the representation MATH needs.
template <int MODE>
struct Acc;
template <>
struct Acc<0> {  // scalar
  float v[8][8];
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) v[i][j] = 0.f;
  }
  __device__ __forceinline__ float get(int i, int j) const { return v[i][j]; }
};
template <>
struct Acc<1> {  // pairs along n: p[i][jp] = (row i, cols 2jp, 2jp+1)
  uint64_t p[8][4];
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) p[i][j] = 0ull;
  }
  __device__ __forceinline__ float get(int i, int j) const {
    const float2 f = unpack2(p[i][j >> 1]);
    return (j & 1) ? f.y : f.x;
  }
};
template <>
struct Acc<2> {  // d[q][r] = (acc(2q,2r), acc(2q+1,2r+1)); e[q][r] = (acc(2q,2r+1), acc(2q+1,2r))
  uint64_t d[4][4], e[4][4];
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int r = 0; r < 4; ++r) { d[q][r] = 0ull; e[q][r] = 0ull; }
  }
  __device__ __forceinline__ float get(int i, int j) const {
    const int q = i >> 1, r = j >> 1;
    const bool ei = i & 1, ej = j & 1;
    if (ei == ej) { const float2 f = unpack2(d[q][r]); return ei ? f.y : f.x; }
    const float2 f = unpack2(e[q][r]);
    return ei ? f.y : f.x;
  }
};

template <bool A_K, bool B_K, bool VEC, bool SPLIT>
__global__ void __launch_bounds__(THREADS, GB300_SG_MIN_BLOCKS) sgemm_ffma_kernel(const Params p) {
  // A held as a row tile only when stored [M,K] and not transposed on the way in
  constexpr bool A_ROWS = A_K && !A_TRANSPOSE;
  constexpr int MODE = (MATH == 2 && A_ROWS) ? 1 : MATH;  // pairs of rows need a k-major A
  extern __shared__ __align__(16) float smem[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int wm = (warp >> 2) * 64;  // warp's first row in the tile
  const int wn = (warp & 3) * 32;   // warp's first column
  const int ty = lane >> 2, tx = lane & 3;
  const int arow = wm + ty * 4;     // lane rows: arow + {0..3}, arow + 32 + {0..3}
  const int bcol = wn + tx * 4;     // lane cols: bcol + {0..3}, bcol + 16 + {0..3}
  const int aswz = (arow >> 2) & 7; // row-tile chunk permutation, shared by all 8 lane rows

  // grouped rasterisation of the tile grid (consecutive blocks share B panels
  // within a group of GROUP_M tile-rows)
  const int bid = blockIdx.x;
  const int per_group = GROUP_M * p.tiles_n;
  const int first_m = (bid / per_group) * GROUP_M;
  const int gsize = min(p.tiles_m - first_m, GROUP_M);
  const int tm = first_m + (bid % per_group) % gsize;
  const int tn = (bid % per_group) / gsize;
  const int m0 = tm * BM, n0 = tn * BN;

  const int kbeg = blockIdx.z * p.k_slice;
  const int kend = min(p.K, kbeg + p.k_slice);
  const int nk = (kend - kbeg + BK - 1) / BK;

  const uint32_t sbase = smem_u32(smem);
  auto stage_load = [&](int s, int k0) {
    const uint32_t st = sbase + (uint32_t)(s * STAGE_FLOATS) * 4u;
    if constexpr (A_ROWS) load_rows<VEC>(st, p.A, p.lda, m0, p.M, k0, kend, tid);
    else if constexpr (A_K) load_transpose(st, p.A, p.lda, m0, p.M, k0, kend, tid);
    else load_kmajor<VEC>(st, p.A, p.lda, m0, p.M, k0, kend, tid);
    const uint32_t sb = st + TILE_FLOATS * 4u;
    if constexpr (B_K) load_transpose(sb, p.B, p.ldb, n0, p.N, k0, kend, tid);
    else load_kmajor<VEC>(sb, p.B, p.ldb, n0, p.N, k0, kend, tid);
  };

  Acc<MODE> acc;
  acc.zero();

#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < nk) stage_load(s, kbeg + s * BK);
    cp_async_commit();
  }

  for (int kt = 0; kt < nk; ++kt) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();  // stage kt visible to all; stage kt-1 fully consumed
    {
      const int nxt = kt + STAGES - 1;
      if (nxt < nk) stage_load(nxt % STAGES, kbeg + nxt * BK);
      cp_async_commit();
    }
    const float* As = smem + (kt % STAGES) * STAGE_FLOATS;
    const float* Bs = As + TILE_FLOATS;
#pragma unroll KC_UNROLL
    for (int kc = 0; kc < BK / 4; ++kc) {
      float a[8][4];  // a[i][kk]: row i, k = 4kc + kk (row-tile A)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const int k = kc * 4 + kk;
        const float* brow = Bs + k * PAD + bcol;
        if constexpr (A_ROWS) {
          // two k at a time (64-bit loads) keeps 16 rather than 32 A values live
          if ((kk & 1) == 0) {
            const float* base = As + arow * BK + ((kc ^ aswz) * 4) + kk;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float2 v = *reinterpret_cast<const float2*>(base + (i < 4 ? i : 32 + i - 4) * BK);
              a[i][kk] = v.x; a[i][kk + 1] = v.y;
            }
          }
        }
        if constexpr (MODE == 2) {
          // k-major A and B: pairs (row 2q, 2q+1) and (col 2r, 2r+1)
          const float* arow_p = As + k * PAD + arow;
          const ulonglong2 a01 = *reinterpret_cast<const ulonglong2*>(arow_p);
          const ulonglong2 a23 = *reinterpret_cast<const ulonglong2*>(arow_p + 32);
          const ulonglong2 b01 = *reinterpret_cast<const ulonglong2*>(brow);
          const ulonglong2 b23 = *reinterpret_cast<const ulonglong2*>(brow + 16);
          const uint64_t ap[4] = {a01.x, a01.y, a23.x, a23.y};
          const uint64_t bp[4] = {b01.x, b01.y, b23.x, b23.y};
          uint64_t bs[4];
#pragma unroll
          for (int r = 0; r < 4; ++r) bs[r] = swap2(bp[r]);
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              acc.d[q][r] = ffma2(ap[q], bp[r], acc.d[q][r]);
              acc.e[q][r] = ffma2(ap[q], bs[r], acc.e[q][r]);
            }
        } else {
          float av[8];
          if constexpr (A_ROWS) {
#pragma unroll
            for (int i = 0; i < 8; ++i) av[i] = a[i][kk];
          } else {
            const float4 lo = lds128(As + k * PAD + arow);
            const float4 hi = lds128(As + k * PAD + arow + 32);
            av[0] = lo.x; av[1] = lo.y; av[2] = lo.z; av[3] = lo.w;
            av[4] = hi.x; av[5] = hi.y; av[6] = hi.z; av[7] = hi.w;
          }
          if constexpr (MODE == 1) {
            const ulonglong2 b01 = *reinterpret_cast<const ulonglong2*>(brow);
            const ulonglong2 b23 = *reinterpret_cast<const ulonglong2*>(brow + 16);
            const uint64_t bp[4] = {b01.x, b01.y, b23.x, b23.y};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint64_t ap = splat2(av[i]);
#pragma unroll
              for (int j = 0; j < 4; ++j) acc.p[i][j] = ffma2(ap, bp[j], acc.p[i][j]);
            }
          } else {
            const float4 b0 = lds128(brow), b1 = lds128(brow + 16);
            const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
              for (int j = 0; j < 8; ++j) acc.v[i][j] = __fmaf_rn(av[i], bv[j], acc.v[i][j]);
          }
        }
      }
    }
  }
  cp_async_wait<0>();

  // epilogue: lane columns bcol + {0..3} and bcol + 16 + {0..3}
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int gm = m0 + arow + (i < 4 ? i : 32 + i - 4);
    if (gm >= p.M) continue;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int gn = n0 + bcol + h * 16;
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = acc.get(i, h * 4 + j);
      if constexpr (SPLIT) {
        float* dst = p.partial + ((int64_t)blockIdx.z * p.M + gm) * p.N + gn;
        if (gn + 3 < p.N && (p.N & 3) == 0) {
          *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (gn + j < p.N) dst[j] = v[j];
        }
      } else {
        float* dst = p.C + (int64_t)gm * p.ldc + gn;
        const bool vec_ok = VEC && (gn + 3 < p.N);
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
          *reinterpret_cast<float4*>(dst) = o;
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (gn + j < p.N) {
              dst[j] = (p.beta != 0.f) ? __fmaf_rn(p.alpha, v[j], p.beta * dst[j])
                                       : p.alpha * v[j];
            }
          }
        }
      }
    }
  }
}

template <bool A_K, bool B_K, bool VEC, bool SPLIT>
cudaError_t launch_one(const Params& p, dim3 grid, cudaStream_t stream) {
  auto kern = sgemm_ffma_kernel<A_K, B_K, VEC, SPLIT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kern<<<grid, THREADS, SMEM_BYTES, stream>>>(p);
  return cudaGetLastError();
}

template <bool A_K, bool B_K>
cudaError_t launch_vs(const Params& p, bool vec, bool split, dim3 grid, cudaStream_t s) {
  if (vec) {
    return split ? launch_one<A_K, B_K, true, true>(p, grid, s)
                 : launch_one<A_K, B_K, true, false>(p, grid, s);
  }
  return split ? launch_one<A_K, B_K, false, true>(p, grid, s)
               : launch_one<A_K, B_K, false, false>(p, grid, s);
}

}  // namespace

cudaError_t launch_sgemm(const SgemmArgs& a, LaunchCtx& ctx) {
  Params p;
  p.A = a.A; p.B = a.B; p.C = a.C; p.partial = a.partial;
  p.lda = a.lda; p.ldb = a.ldb; p.ldc = a.ldc;
  p.M = a.M; p.N = a.N; p.K = a.K;
  p.k_slice = a.splits > 1 ? a.k_slice : a.K;
  p.tiles_m = (a.M + BM - 1) / BM;
  p.tiles_n = (a.N + BN - 1) / BN;
  p.alpha = a.alpha; p.beta = a.beta;
  // 16-byte staging needs 16-byte aligned rows in every operand (C too: the
  // epilogue's float4 accesses share the flag).
  const bool vec = ((reinterpret_cast<uintptr_t>(a.A) | reinterpret_cast<uintptr_t>(a.B) |
                     reinterpret_cast<uintptr_t>(a.C)) & 15u) == 0 &&
                   (a.lda % 4) == 0 && (a.ldb % 4) == 0 && (a.ldc % 4) == 0;
  const bool split = a.splits > 1;
  dim3 grid(p.tiles_m * p.tiles_n, 1, split ? a.splits : 1);
  const bool A_K = !a.transA, B_K = a.transB;
  cudaError_t e;
  if (A_K && !B_K) e = launch_vs<true, false>(p, vec, split, grid, ctx.stream);
  else if (!A_K && !B_K) e = launch_vs<false, false>(p, vec, split, grid, ctx.stream);
  else if (A_K && B_K) e = launch_vs<true, true>(p, vec, split, grid, ctx.stream);
  else e = launch_vs<false, true>(p, vec, split, grid, ctx.stream);
  if (e == cudaSuccess) ctx.launches++;
  return e;
}

}  // namespace gb300
