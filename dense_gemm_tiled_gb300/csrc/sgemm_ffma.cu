// FP32 SGEMM on the CUDA cores: C = alpha * op(A) * op(B) + beta * C.
//
// What the pages contribute (design ideas, not code):
//  - "Optimizing GEMM on Apple's M5 from scratch, Part 1": shared-memory
//    tiling (kernels 2-3: every input tile is loaded once per block and reused
//    by all its threads) and thread coarsening (kernel 4: one thread owns
//    several outputs so an operand value held in a register feeds several
//    FMAs).  Here the coarsening is two-dimensional, an 8 x 8 register block
//    per thread, the register blocking of "From a C loop to a GPU kernel"
//    ("Register blocking" and its 2x2 -> 4x4 -> 8x8 plan).
//  - "From a C loop to a GPU kernel", "Double buffering": the next K tile is
//    fetched while the current one is consumed.  Here a 4-stage cp.async ring.
//  - "Metal GEMM Kernels for LoRA Training", section 3: the transposed
//    operand cost instruction count, not memory traffic.  Here no operand is
//    transposed in memory at all: each operand is staged in the orientation it
//    is stored in, and the inner loop reads it with 128-bit shared loads along
//    whichever dimension is contiguous (k for A[M,K] / B[N,K]; m or n for
//    A[K,M] / B[K,N]).
//  - "Part 1", kernel 1: consecutive threads own consecutive columns, so
//    global loads are coalesced; here every global load is a 16-byte cp.async
//    and a warp's loads cover whole 64- or 512-byte row segments.
//
// Tile: 128 x 128 outputs per block, K step 16, 256 threads (8 warps as 2 x 4,
// each warp 64 x 32, each lane 8 x 8 outputs split into 4-wide groups).
// Arithmetic is IEEE fp32 FMA (__fmaf_rn), no fast-math, denormals kept.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace gb300 {
namespace {

constexpr int BM = SG_BM, BN = SG_BN, BK = SG_BK;
constexpr int STAGES = 4;
constexpr int THREADS = 256;
constexpr int TILE_FLOATS = BM * BK;  // per operand per stage (BM == BN)
constexpr int STAGE_FLOATS = 2 * TILE_FLOATS;
constexpr int SMEM_BYTES = STAGES * STAGE_FLOATS * 4;  // 64 KiB
constexpr int GROUP_M = 8;  // tile rasterisation: 8 tile-rows walked together

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

// Operand staging.  An operand is "K-contiguous" when k is its fastest index
// (A stored [M,K], B stored [N,K]) and "MN-contiguous" otherwise.
//  K-contiguous tile  : 128 rows (m or n) x 16 k, 64 bytes a row, the four
//                       16-byte chunks of a row permuted by chunk ^ ((row>>2)&3)
//                       so the 128-bit fragment reads of a warp hit distinct
//                       banks.
//  MN-contiguous tile : 16 rows (k) x 128 (m or n), 512 bytes a row.
__device__ __forceinline__ int kc_swz(int row, int chunk) { return chunk ^ ((row >> 2) & 3); }

template <bool KCONTIG, bool VEC>
__device__ __forceinline__ void load_tile(uint32_t dst, const float* __restrict__ g, int64_t ld,
                                          int mn0, int MN, int k0, int K, int tid) {
  if constexpr (VEC) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int q = tid + r * THREADS;
      if constexpr (KCONTIG) {
        const int row = q >> 2, c = q & 3;
        const int gm = mn0 + row, gk = k0 + c * 4;
        const bool ok = (gm < MN) && (gk < K);
        const uint32_t bytes = ok ? (uint32_t)min(4, K - gk) * 4u : 0u;
        const float* src = ok ? g + (int64_t)gm * ld + gk : g;
        cp_async_16(dst + (uint32_t)(row * BK + kc_swz(row, c) * 4) * 4u, src, bytes);
      } else {
        const int krow = q >> 5, c = q & 31;
        const int gk = k0 + krow, gm = mn0 + c * 4;
        const bool ok = (gk < K) && (gm < MN);
        const uint32_t bytes = ok ? (uint32_t)min(4, MN - gm) * 4u : 0u;
        const float* src = ok ? g + (int64_t)gk * ld + gm : g;
        cp_async_16(dst + (uint32_t)(krow * BM + c * 4) * 4u, src, bytes);
      }
    }
  } else {
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int e = tid + r * THREADS;
      if constexpr (KCONTIG) {
        const int row = e >> 4, kk = e & 15;
        const int gm = mn0 + row, gk = k0 + kk;
        const bool ok = (gm < MN) && (gk < K);
        const float* src = ok ? g + (int64_t)gm * ld + gk : g;
        const int col = kc_swz(row, kk >> 2) * 4 + (kk & 3);
        cp_async_4(dst + (uint32_t)(row * BK + col) * 4u, src, ok ? 4u : 0u);
      } else {
        const int krow = e >> 7, mm = e & 127;
        const int gk = k0 + krow, gm = mn0 + mm;
        const bool ok = (gk < K) && (gm < MN);
        const float* src = ok ? g + (int64_t)gk * ld + gm : g;
        cp_async_4(dst + (uint32_t)(krow * BM + mm) * 4u, src, ok ? 4u : 0u);
      }
    }
  }
}

__device__ __forceinline__ float4 lds128(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}

// Fragment for 4 consecutive k (k = kc*4 .. kc*4+3) of this lane's 8 rows
// (m or n): frag[i][kk].  `base` is the lane's first row inside the tile;
// rows are base + {0,1,2,3} and base + HALF + {0,1,2,3}.
template <bool KCONTIG, int HALF>
__device__ __forceinline__ void load_frag_k4(float (&frag)[8][4], const float* tile, int base,
                                             int kc) {
  if constexpr (KCONTIG) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int row = base + (i < 4 ? i : HALF + i - 4);
      const float4 v = lds128(tile + row * BK + kc_swz(row, kc) * 4);
      frag[i][0] = v.x; frag[i][1] = v.y; frag[i][2] = v.z; frag[i][3] = v.w;
    }
  } else {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const float* rowp = tile + (kc * 4 + kk) * BM;
      const float4 lo = lds128(rowp + base);
      const float4 hi = lds128(rowp + base + HALF);
      frag[0][kk] = lo.x; frag[1][kk] = lo.y; frag[2][kk] = lo.z; frag[3][kk] = lo.w;
      frag[4][kk] = hi.x; frag[5][kk] = hi.y; frag[6][kk] = hi.z; frag[7][kk] = hi.w;
    }
  }
}

template <bool A_K, bool B_K, bool VEC, bool SPLIT>
__global__ void __launch_bounds__(THREADS, (A_K && B_K) ? 1 : 2)
    sgemm_ffma_kernel(const Params p) {
  extern __shared__ __align__(16) float smem[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int wm = (warp >> 2) * 64;  // warp's first row in the tile
  const int wn = (warp & 3) * 32;   // warp's first column
  const int ty = lane >> 2, tx = lane & 3;
  const int arow = wm + ty * 4;     // lane rows: arow + {0..3}, arow + 32 + {0..3}
  const int bcol = wn + tx * 4;     // lane cols: bcol + {0..3}, bcol + 16 + {0..3}

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
  // A operand rows run along m, B operand "rows" along n.
  auto stage_load = [&](int s, int k0) {
    const uint32_t st = sbase + (uint32_t)(s * STAGE_FLOATS) * 4u;
    load_tile<A_K, VEC>(st, p.A, p.lda, m0, p.M, k0, kend, tid);
    load_tile<B_K, VEC>(st + TILE_FLOATS * 4u, p.B, p.ldb, n0, p.N, k0, kend, tid);
  };

  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

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
#pragma unroll
    for (int kc = 0; kc < BK / 4; ++kc) {
      float a[8][4], b[8][4];
      load_frag_k4<A_K, 32>(a, As, arow, kc);
      load_frag_k4<B_K, 16>(b, Bs, bcol, kc);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i][j] = __fmaf_rn(a[i][kk], b[j][kk], acc[i][j]);
    }
  }
  cp_async_wait<0>();

  // epilogue
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int gm = m0 + arow + (i < 4 ? i : 32 + i - 4);
    if (gm >= p.M) continue;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int gn = n0 + bcol + h * 16;
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = acc[i][h * 4 + j];
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
