#pragma once
// 16-bit-operand (fp16 or bf16) / fp32-accumulate / 16-bit-output GEMM on the
// 5th-generation tensor cores (tcgen05.mma, accumulators in tensor memory).
// This header holds the kernel and its launcher templated on the element type;
// hgemm_tcgen05.cu instantiates them for fp16 (and holds the dispatcher's
// planning functions), hgemm_bf16.cu for bf16.
//
//   C = alpha * op(A) * op(B) + beta * C, variants nn / tn / nt (and tt).
//
// The regime is that of "Metal GEMM Kernels for LoRA Training on Apple
// Silicon": fp16 operands with fp32 accumulation (section 1, type table), the
// fp32 accumulator converted to fp16 on the way out (section 2), the three
// transpose variants of the section 2 table, and fp32 partial sums plus a
// reduction for skinny shapes (section 5, split-K).  The Metal design there (one
// 32 x 32 simdgroup tile, staged output) is prior art only; this kernel is
// built for sm_103a:
//
//  * Persistent, warp-specialised block of 6 warps, one block per SM:
//      warp 0      TMA producer (one elected lane)
//      warp 1      TMEM allocator + MMA issuer (one elected lane)
//      warps 2..5  epilogue (128 threads = the 128 accumulator rows)
//  * Operand tiles reach shared memory by TMA (cp.async.bulk.tensor) with the
//    128-byte swizzle, through a ring of STAGES buffers guarded by mbarriers
//    (full: TMA bytes landed; empty: the MMAs reading the buffer finished).
//    Out-of-range rows/columns of edge tiles are zero-filled by the TMA unit.
//  * The transposed operand is not moved: a K-contiguous operand (A[M,K],
//    B[N,K]) is described to the tensor core as K-major, an MN-contiguous one
//    (A[K,M], B[K,N]) as MN-major, by the shared-memory descriptor layout and
//    the instruction descriptor's major bits.  Section 3 of the LoRA page
//    found the transposed operand's cost in staging instructions; here there
//    are none.
//  * The 128 x BN fp32 accumulator lives in tensor memory, double buffered,
//    so the epilogue of one tile overlaps the main loop of the next.
//  * Fused epilogue: tcgen05.ld -> alpha * acc + beta * C_old -> fp16
//    (round to nearest even) -> TMA store through swizzled staging.
//  * Schedule: whole tiles round-robin over the persistent grid, optionally
//    followed by stream-K -- the K steps of the last tiles shared out in equal
//    contiguous ranges, a tile shared by several ranges finished by its last
//    contributor from the others' fp32 partial sums (section 5's split-K,
//    with the reduction inside the GEMM kernel and no waiting between blocks).
//
// Every mbarrier wait is bounded (see common.cuh); on expiry the block stops
// issuing work, drains its in-flight copies and MMAs, frees its tensor memory
// and returns, leaving GEMM_ERR_TIMEOUT in the device status word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <type_traits>

#include "common.cuh"
#include "internal.h"
#include "tensor_map.h"

namespace gb300 {
namespace {

// The 16-bit operand/output types of kind::f16 MMAs: IEEE binary16 and
// bfloat16 (same tensor-core rate; they differ in the instruction
// descriptor's A/B format field, the TMA element type and the output cast).
template <typename T>
struct Elem;
template <>
struct Elem<__half> {
  using T2 = __half2;
  static constexpr uint32_t FMT = 0;  // kind::f16 A/B format: F16
  static constexpr CUtensorMapDataType TMA = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  static __device__ __forceinline__ T2 pack(float a, float b) { return __floats2half2_rn(a, b); }
  static __device__ __forceinline__ float2 unpack(T2 v) { return __half22float2(v); }
  static __device__ __forceinline__ __half from(float f) { return __float2half_rn(f); }
  static __device__ __forceinline__ float to(__half v) { return __half2float(v); }
};
template <>
struct Elem<__nv_bfloat16> {
  using T2 = __nv_bfloat162;
  static constexpr uint32_t FMT = 1;  // kind::f16 A/B format: BF16
  static constexpr CUtensorMapDataType TMA = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  static __device__ __forceinline__ T2 pack(float a, float b) { return __floats2bfloat162_rn(a, b); }
  static __device__ __forceinline__ float2 unpack(T2 v) { return __bfloat1622float2(v); }
  static __device__ __forceinline__ __nv_bfloat16 from(float f) { return __float2bfloat16_rn(f); }
  static __device__ __forceinline__ float to(__nv_bfloat16 v) { return __bfloat162float(v); }
};

// fp32 operands for the opt-in TF32 path (kind::tf32; output fp32)
template <>
struct Elem<float> {
  using T2 = float2;
  static constexpr uint32_t FMT = 2;  // kind::tf32 A/B format: TF32
  static constexpr CUtensorMapDataType TMA = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  static __device__ __forceinline__ T2 pack(float a, float b) { return make_float2(a, b); }
  static __device__ __forceinline__ float2 unpack(T2 v) { return v; }
  static __device__ __forceinline__ float from(float f) { return f; }
  static __device__ __forceinline__ float to(float v) { return v; }
};

// Elements of T in one 128-byte swizzle-atom row: the K depth of a stage (64
// for 16-bit operands, 32 for fp32), and the K of one MMA (32 bytes: 16 or 8).
template <typename T>
__host__ __device__ constexpr int kblk() { return 128 / (int)sizeof(T); }
template <typename T>
__host__ __device__ constexpr int kmma() { return 32 / (int)sizeof(T); }

constexpr int BM = HG_BM;     // 128 accumulator rows = 128 TMEM lanes
constexpr int BK = HG_BK;     // 64 fp16 = 128 bytes = one swizzle atom row (16-bit types)
// Epilogue warps: 4 (one per 32-lane quarter of the accumulator) or 8 (two per
// quarter, each draining half of the tile's columns)
#ifndef GB300_HG_EPI_WARPS
#define GB300_HG_EPI_WARPS 8
#endif
constexpr int EPI_WARPS = GB300_HG_EPI_WARPS;
constexpr int EPI_HALVES = EPI_WARPS / 4;
static_assert(EPI_WARPS == 4 || EPI_WARPS == 8, "epilogue warps");
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr int GROUP_M = 8;
constexpr int A_TILE_BYTES = BM * BK * 2;  // 16 KiB
constexpr int SMEM_LIMIT = 227 * 1024;  // opt-in shared memory per block

// MODE: 0 = single blocks; 2 = pairs running 256-row MMAs across both SMs
// (tcgen05 cta_group::2): each block holds its 128 rows of A and half of the
// B tile.
template <int BN, bool B_MN, int MODE = 0>
struct Cfg {
  static_assert(MODE == 0 || MODE == 2, "kernel mode");
  // An MN-major B tile is stored as 64-wide swizzle atoms, so it is at least
  // one atom wide; the MMA reads only the first BN columns.
  static constexpr int B_COLS = B_MN ? (BN < 64 ? 64 : BN) : BN;
  static constexpr int B_TILE_BYTES = (MODE == 2 ? B_COLS / 2 : B_COLS) * BK * 2;
  static constexpr int STAGE_BYTES = A_TILE_BYTES + B_TILE_BYTES;
  // C staging for TMA stores: 4 KiB buffers (one 32-row box of 128-byte rows).
  // Four epilogue warps take two each when that costs no pipeline stage, else
  // one; eight warps (both column shares, for short-K tiles) take one each and
  // are allowed only where that costs no stage either (EPI2).
  static constexpr int FIXED_BYTES = 1024 /*align*/ + 512 /*barriers*/;
  static constexpr int STAGES_OF(int staging) {
    return (SMEM_LIMIT - FIXED_BYTES - staging) / STAGE_BYTES;
  }
  static constexpr int NBUF4 = (STAGES_OF(8 * 4096) >= 8 || STAGES_OF(8 * 4096) == STAGES_OF(4 * 4096)) ? 2 : 1;
  static constexpr int STAGING4 = 4 * NBUF4 * 4096;
  static constexpr bool EPI2 = EPI_WARPS == 8 && STAGES_OF(8 * 4096) >= (STAGES_OF(STAGING4) < 8 ? STAGES_OF(STAGING4) : 8);
  static constexpr int STAGING_BYTES = (EPI2 && STAGING4 < 8 * 4096) ? 8 * 4096 : STAGING4;
  static constexpr int STAGES_RAW = STAGES_OF(STAGING_BYTES);
  static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
  // two accumulator buffers of BN fp32 columns, rounded up to a power of two
  static constexpr int TMEM_COLS = 2 * BN <= 64 ? 64 : 2 * BN <= 128 ? 128 : 2 * BN <= 256 ? 256 : 512;
  static constexpr int SMEM_BYTES =
      STAGES * STAGE_BYTES + STAGING_BYTES + FIXED_BYTES;
};

struct HParams {
  void* C;  // __half, __nv_bfloat16 or float, per the kernel's element type
  int64_t ldc;
  int M, N, K;
  int tiles_m, tiles_n;  // 128-row tiles and BN-column tiles of one matrix
  // Work tiles: one per (batch entry, row of tiles -- a row of tile pairs
  // with pairs --, column of tiles), `steps` K steps of kblk each.
  int tiles, steps;
  // Schedule (a persistent grid of W workers: blocks, or block pairs):
  //  * tiles [0, dp_tiles) are whole units, worker w taking w, w + W, ...;
  //  * the K steps of the other tiles, (tiles - dp_tiles) * steps of them in
  //    tile-major order, are cut into sk_workers contiguous ranges of (almost)
  //    equal length, worker w < sk_workers taking range w (stream-K).  A range
  //    covers the end of one tile, whole tiles, and the start of another; a
  //    tile covered by one range is stored as usual, a tile shared by several
  //    ranges is finished by whichever contributor arrives last (below).
  int dp_tiles, sk_workers;
  int64_t sk_steps;
  // floor((2^64 - 1) / d) for d = sk_workers, sk_steps, steps (div_magic)
  uint64_t m_skw, m_sks, m_steps;
  // 3xTF32: a tile's steps are its steps_k K steps three times over, step g
  // reading K step g / 3 of the (A plane, B plane) pair (hi, hi), (hi, lo),
  // (lo, hi) for g % 3 = 0, 1, 2; the planes are the operand maps' third
  // coordinate
  int split3, steps_k;
  // Shared tiles: each contributing range writes its fp32 partial sums to its
  // slot of sk_ws -- [sk_workers][2: the range's first / last tile][pair ? 2 :
  // 1][4 lane quarters][32 x BN], each quarter's strip laid out as one warp
  // holds it ([32-column chunk][float4][lane]) -- then counts itself in
  // sk_cnt[shared tile][pair ? 2 : 1][4][EPI_HALVES] (zero at launch); the
  // last to count sums every contributor's slot in K order, runs the epilogue
  // and puts the counter back to zero.  No block waits for another.
  float* sk_ws;
  unsigned int* sk_cnt;
  // 1: every contributor only publishes its partial sums and a separate
  // reduction kernel (hgemm_sk_reduce) finishes the shared tiles; sk_cnt unused
  int sk_publish;
  float alpha, beta;
  unsigned int* status;
  uint64_t timeout_ns;
  int fault_injection;
  int c_vec_ok;  // C base 16-byte aligned and ldc % (16 / element size) == 0
  int c_tma;     // C aligned: C leaves through TMA stores (and comes in by TMA loads)
  int pair;      // 2: clusters of two blocks run 2-SM (cta_group::2) MMAs; 0: single blocks
  // strided batch: the tensor maps carry the batch entry as their third
  // coordinate
  int batch;
  int64_t stride_c;  // elements between consecutive C matrices
  int za_mask, zb_mask;  // -1: operand batched; 0: one matrix shared by all (pitch 0)
  Epilogue ep;           // bias (output type, per column) and activation
  int epi_halves;        // epilogue warps in use per accumulator quarter: 1 or EPI_HALVES
};

// tcgen05 shared-memory matrix descriptor, 128-byte swizzle:
//   bits  0-13  start address >> 4
//   bits 16-29  leading-dimension byte offset >> 4
//   bits 32-45  stride-dimension byte offset >> 4
//   bits 46-48  fixed 0b001
//   bits 61-63  layout: 2 = 128-byte swizzle
// K-major:  rows of 128 B (64 fp16 along K), 8-row groups 1024 B apart (SBO);
//           the leading offset is unused for a swizzled K-major operand.
// MN-major: rows of 128 B (64 fp16 along M or N) indexed by k; 8-k-row groups
//           1024 B apart (SBO); 64-wide M/N atoms BK*128 B apart (LBO).
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B format
// (bits 7-9, 10-12: 0 fp16, 1 bf16), A major (bit 15), B major (bit 16;
// 1 = MN-major), N >> 3 (bits 17-22), M >> 4 (bits 24-28).
template <int BN, bool A_MN, bool B_MN, int M_ROWS = BM, uint32_t FMT = 0>
__device__ __forceinline__ constexpr uint32_t make_idesc() {
  return (1u << 4) | (FMT << 7) | (FMT << 10) | ((A_MN ? 1u : 0u) << 15) |
         ((B_MN ? 1u : 0u) << 16) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(M_ROWS >> 4) << 24);
}

// One unit of a worker's work: this block's 128 rows of a tile (from m0),
// its columns from n0, batch entry bz, K steps [kb0, kb0 + nkb).  sk >= 0
// marks a shared tile (stream-K tile sk, counted from dp_tiles) whose partial
// sums from this range go to the range's slot `slot`.  Without pairs a tile is
// 128 x BN; with pairs a tile is two vertically adjacent 128-row tiles and
// block `rank` of the pair takes tile row 2 * pair_row + rank.
struct Unit {
  int m0, n0, bz, kb0, nkb, sk, slot;
};

// First stream-K step of range w (range w is [sk_begin(w), sk_begin(w + 1))).
__device__ __forceinline__ int64_t sk_begin(const HParams& p, int w) {
  return (int64_t)div_magic((uint64_t)w * (uint64_t)p.sk_steps, (uint64_t)p.sk_workers, p.m_skw);
}
// The range that holds stream-K step x: the largest w with sk_begin(w) <= x.
__device__ __forceinline__ int sk_owner(const HParams& p, int64_t x) {
  return (int)div_magic((uint64_t)(x + 1) * (uint64_t)p.sk_workers - 1u, (uint64_t)p.sk_steps,
                        p.m_sks);
}
// Slot of range w in shared tile sk: 0 if the range starts in the tile (it is
// the range's first tile), 1 if it started before (its last).
// (sk_begin(w) >= s0 exactly when w * sk_steps >= s0 * sk_workers)
__device__ __forceinline__ int sk_slot(const HParams& p, int w, int64_t s0) {
  return (int64_t)w * p.sk_steps >= s0 * p.sk_workers ? 0 : 1;
}

// Work tile t -> batch entry bz, then grouped rasterisation within the
// entry: block `rank`'s first row m0 and the tile's first column n0.
template <bool PAIR, int TBN>
__device__ __forceinline__ void tile_origin(const HParams& p, int t, int rank, int& m0, int& n0,
                                            int& bz) {
  const int rows = PAIR ? (p.tiles_m + 1) / 2 : p.tiles_m;
  const int per_entry = rows * p.tiles_n;
  bz = t / per_entry;
  t -= bz * per_entry;
  const int per_group = GROUP_M * p.tiles_n;
  const int first_m = (t / per_group) * GROUP_M;
  const int gsize = min(rows - first_m, GROUP_M);
  const int tr = first_m + (t % per_group) % gsize;
  const int tn = (t % per_group) / gsize;
  const int tm = PAIR ? 2 * tr + rank : tr;
  m0 = tm * BM;
  n0 = tn * TBN;
}

// Unit i of worker w (of W); false when the worker has no unit i.  Every role
// of the block walks the same sequence: the worker's whole tiles first, then
// the tiles its stream-K range touches, in K order.
template <bool PAIR, int TBN>
__device__ __forceinline__ bool unit_at(const HParams& p, int w, int W, int i, int rank,
                                        Unit& u) {
  const int n_dp = w < p.dp_tiles ? (p.dp_tiles - 1 - w) / W + 1 : 0;
  int t;
  u.kb0 = 0;
  u.nkb = p.steps;
  u.sk = -1;
  u.slot = 0;
  if (i < n_dp) {
    t = w + i * W;
  } else {
    if (w >= p.sk_workers) return false;
    const int64_t b = sk_begin(p, w), e = sk_begin(p, w + 1);
    const int64_t tr = (int64_t)div_magic((uint64_t)b, (uint64_t)p.steps, p.m_steps) + (i - n_dp);
    const int64_t s0 = tr * p.steps;
    const int64_t lo = b > s0 ? b : s0;
    const int64_t hi = e < s0 + p.steps ? e : s0 + p.steps;
    if (hi <= lo) return false;
    u.kb0 = (int)(lo - s0);
    u.nkb = (int)(hi - lo);
    if (u.nkb < p.steps) {
      u.sk = (int)tr;
      u.slot = b >= s0 ? 0 : 1;  // the range's first tile, or its last
    }
    t = p.dp_tiles + (int)tr;
  }
  tile_origin<PAIR, TBN>(p, t, rank, u.m0, u.n0, u.bz);
  return true;
}

// act(alpha * v + beta * C + bias) -> T (RN-even) -> C, for 32 columns of one
// row (every loop fully unrolled, so v stays in registers)
template <typename T>
__device__ __forceinline__ void store_c32(const HParams& p, int bz, int gm, int gn0,
                                          float (&v)[32]) {
  using E = Elem<T>;
  T* dst = static_cast<T*>(p.C) + (int64_t)bz * p.stride_c + (int64_t)gm * p.ldc + gn0;
  const bool full = (gn0 + 31 < p.N) && p.c_vec_ok;
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = p.alpha * v[j];
  if (p.beta != 0.f) {
    if (!full) {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (gn0 + j < p.N) v[j] = __fmaf_rn(p.beta, E::to(dst[j]), v[j]);
    } else if constexpr (sizeof(T) == 4) {
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const float4 cv = reinterpret_cast<const float4*>(dst)[w];
        v[4 * w] = __fmaf_rn(p.beta, cv.x, v[4 * w]);
        v[4 * w + 1] = __fmaf_rn(p.beta, cv.y, v[4 * w + 1]);
        v[4 * w + 2] = __fmaf_rn(p.beta, cv.z, v[4 * w + 2]);
        v[4 * w + 3] = __fmaf_rn(p.beta, cv.w, v[4 * w + 3]);
      }
    } else {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const uint4 cv = reinterpret_cast<const uint4*>(dst)[w];
        const typename E::T2* ch = reinterpret_cast<const typename E::T2*>(&cv);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = E::unpack(ch[e]);
          v[8 * w + 2 * e] = __fmaf_rn(p.beta, f.x, v[8 * w + 2 * e]);
          v[8 * w + 2 * e + 1] = __fmaf_rn(p.beta, f.y, v[8 * w + 2 * e + 1]);
        }
      }
    }
  }
  if (p.ep.bias != nullptr || p.ep.act != 0) {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (gn0 + j < p.N) v[j] = apply_epilogue<T>(v[j], p.ep, gn0 + j);
  }
  if (!full) {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (gn0 + j < p.N) dst[j] = E::from(v[j]);
  } else if constexpr (sizeof(T) == 4) {
#pragma unroll
    for (int w = 0; w < 8; ++w)
      reinterpret_cast<float4*>(dst)[w] =
          make_float4(v[4 * w], v[4 * w + 1], v[4 * w + 2], v[4 * w + 3]);
  } else {
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint4 o;
      typename E::T2* oh = reinterpret_cast<typename E::T2*>(&o);
#pragma unroll
      for (int e = 0; e < 4; ++e) oh[e] = E::pack(v[8 * w + 2 * e], v[8 * w + 2 * e + 1]);
      reinterpret_cast<uint4*>(dst)[w] = o;
    }
  }
}

// The same for a 32 x 32 block of C (rows gm0 .., columns gn0 ..; lane l holds
// row gm0 + l in r) whose rows are not 16-byte aligned, through this warp's
// 4 KiB staging buffer: row by row from lane-owned rows, every global access
// of the warp touches 32 rows (measured 4095^3 fp16: the kernel at 2.3x the
// time of 4096^3); staged, the block is written in row = lane order (16-byte
// chunk w of row l at chunk w ^ (l & 7), conflict-free) and read back one
// column a lane, so each access covers one row.  C is loaded sixteen rows at
// a time ahead of use.
template <typename T>
__device__ __forceinline__ void store_c32_staged(const HParams& p, int bz, int gm0, int gn0,
                                                 uint32_t sbuf, const uint32_t (&r)[32],
                                                 int lane) {
  using E = Elem<T>;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const uint32_t a = sbuf + (uint32_t)(lane * 128 + ((w ^ (lane & 7)) * 16));
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(r[4 * w]),
                 "r"(r[4 * w + 1]), "r"(r[4 * w + 2]), "r"(r[4 * w + 3])
                 : "memory");
  }
  __syncwarp();
  const bool epi = p.ep.bias != nullptr || p.ep.act != 0;
  const int col = gn0 + lane;
  T* const Cc = static_cast<T*>(p.C) + (int64_t)bz * p.stride_c + (int64_t)gm0 * p.ldc + col;
  const int rows = min(32, p.M - gm0);
#pragma unroll 1
  for (int r0 = 0; r0 < rows; r0 += 16) {
    float cv[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      cv[i] = (p.beta != 0.f && col < p.N && r0 + i < rows) ? E::to(Cc[(int64_t)(r0 + i) * p.ldc])
                                                             : 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int rr = r0 + i;
      if (rr >= rows || col >= p.N) continue;
      float x;
      const uint32_t a =
          sbuf + (uint32_t)(rr * 128 + (((lane >> 2) ^ (rr & 7)) * 16) + (lane & 3) * 4);
      asm volatile("ld.shared.f32 %0, [%1];" : "=f"(x) : "r"(a) : "memory");
      float o = p.alpha * x;
      if (p.beta != 0.f) o = __fmaf_rn(p.beta, cv[i], o);
      if (epi) o = apply_epilogue<T>(o, p.ep, col);
      Cc[(int64_t)rr * p.ldc] = E::from(o);
    }
  }
  __syncwarp();  // the buffer is rewritten by the next block
}

template <typename T, int BN, bool A_MN, bool B_MN, int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    hgemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const HParams p) {
  constexpr bool PAIR = MODE != 0;
  constexpr bool TWO_SM = MODE == 2;
  using C_ = Cfg<BN, B_MN, MODE>;
  constexpr int STAGES = C_::STAGES;
  // bytes that complete one stage: this block's (single), or both blocks'
  // (2-SM pair: all loads of the pair complete on the even block's barrier)
  constexpr uint32_t STAGE_TX = (uint32_t)C_::STAGE_BYTES * (TWO_SM ? 2u : 1u);
  // 2-SM pairs: the even block issues every MMA and its commits arrive on
  // both blocks' barriers.
  const int rank = PAIR ? (int)cluster_ctarank() : 0;
  const int worker = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int workers = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t tiles_addr = (raw_addr + 1023u) & ~1023u;  // swizzle atoms need 1 KiB alignment
  uint8_t* const tiles_ptr = smem_raw + (tiles_addr - raw_addr);
  // C staging (1 KiB aligned: the 128-byte swizzle pattern repeats every 1 KiB)
  const uint32_t staging_addr = tiles_addr + (uint32_t)(STAGES * C_::STAGE_BYTES);
  uint8_t* const staging_ptr = tiles_ptr + STAGES * C_::STAGE_BYTES;
  uint64_t* const bars = reinterpret_cast<uint64_t*>(staging_ptr + C_::STAGING_BYTES);
  // barrier layout: full[STAGES], empty[STAGES], acc_full[2], acc_empty[2], drain,
  // the tensor-memory address slot (and abort flag) ...
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * (uint32_t)s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (uint32_t)(STAGES + s); };
  auto accf_bar = [&](int b) { return bar0 + 8u * (uint32_t)(2 * STAGES + b); };
  auto acce_bar = [&](int b) { return bar0 + 8u * (uint32_t)(2 * STAGES + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (uint32_t)(2 * STAGES + 4);
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
  // ... then one per C staging buffer: its TMA load of C (beta != 0) completed
  constexpr int NSTAGING = C_::STAGING_BYTES / 4096;
  static_assert(8 * (2 * STAGES + 6 + NSTAGING + EPI_WARPS) <= 512, "barrier area");
  auto cload_bar = [&](int b) { return bar0 + 8u * (uint32_t)(2 * STAGES + 6 + b); };
  // ... then one per epilogue warp: its bulk loads of shared-tile partial
  // sums (into the stage ring, once the ring is idle) completed
  auto fix_bar = [&](int w) { return bar0 + 8u * (uint32_t)(2 * STAGES + 6 + NSTAGING + w); };
  volatile uint32_t* const abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf_bar(b), 1);
      // 2-SM pairs: both blocks' epilogues release the accumulator to the
      // even block's MMA issuer
      mbar_init(acce_bar(b), (TWO_SM ? 2 : 1) * 32 * 4 * p.epi_halves);
    }
    mbar_init(drain_bar, 1);
    for (int b = 0; b < NSTAGING; ++b) mbar_init(cload_bar(b), 1);
    for (int w = 0; w < EPI_WARPS; ++w) mbar_init(fix_bar(w), 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    if constexpr (TWO_SM) {
      tmem_alloc_pair(smem_u32(tmem_slot), (uint32_t)C_::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), (uint32_t)C_::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  if constexpr (PAIR) cluster_sync();  // the peer's barriers exist before any remote arrive
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // (set-up above may overlap the previous kernel in the stream; it completes
  // before any global access below)
  pdl_wait();
  pdl_trigger();

  const WaitCtl wc{p.status, abort_flag, p.timeout_ns};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t pending = 0, pend_phase = 0;  // per-stage: last load issued / its parity
      bool first = true;
      bool ok = true;
      Unit U;
      for (int i = 0; ok && unit_at<PAIR, BN>(p, worker, workers, i, rank, U); ++i) {
        const int m0 = U.m0, n0 = U.n0;
        int za = U.bz & p.za_mask, zb = U.bz & p.zb_mask;
        for (int kb = 0; kb < U.nkb; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, wc)) { ok = false; break; }
          int k0 = (U.kb0 + kb) * kblk<T>();
          if (p.split3) {
            // step g is segment g % 3 of K step g / 3: the three products of a
            // K step follow each other, so each plane tile's second use finds
            // it in L2 (segment after segment re-read the planes from DRAM:
            // 2.3 GB a launch at 4096^3)
            const int g = U.kb0 + kb, seg = g % 3;
            k0 = (g / 3) * kblk<T>();
            za = seg == 2 ? 1 : 0;
            zb = seg == 1 ? 1 : 0;
          }
          const bool skip = first && p.fault_injection == 1;
          first = false;
          if (!skip && TWO_SM) {
            // this block's 128 rows of A and half of B, into its own shared
            // memory, completing on the even block's `full` barrier
            const uint32_t sa = tiles_addr + (uint32_t)(stage * C_::STAGE_BYTES);
            const uint32_t sb = sa + (uint32_t)A_TILE_BYTES;
            const uint32_t fb = mapa_shared(full_bar(stage), 0u);
            if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), STAGE_TX);
            if constexpr (A_MN) {
              tma_load_3d_pair(sa, &tmA, m0, k0, za, fb);
              tma_load_3d_pair(sa + 8192u, &tmA, m0 + 64, k0, za, fb);
            } else {
              tma_load_3d_pair(sa, &tmA, k0, m0, za, fb);
            }
            if constexpr (B_MN) {
              constexpr int MINE = (C_::B_COLS / 64) / 2;
#pragma unroll
              for (int h = 0; h < MINE; ++h)
                tma_load_3d_pair(sb + (uint32_t)h * 8192u, &tmB, n0 + 64 * (rank * MINE + h), k0, zb, fb);
            } else {
              tma_load_3d_pair(sb, &tmB, k0, n0 + rank * (BN / 2), zb, fb);
            }
            if (rank == 0) {
              pending |= 1u << stage;
              pend_phase = (pend_phase & ~(1u << stage)) | (phase << stage);
            }
          } else if (!skip) {
            const uint32_t sa = tiles_addr + (uint32_t)(stage * C_::STAGE_BYTES);
            const uint32_t sb = sa + (uint32_t)A_TILE_BYTES;
            mbar_arrive_expect_tx(full_bar(stage), STAGE_TX);
            if constexpr (A_MN) {
              tma_load_3d(sa, &tmA, m0, k0, za, full_bar(stage));
              tma_load_3d(sa + 8192u, &tmA, m0 + 64, k0, za, full_bar(stage));
            } else {
              tma_load_3d(sa, &tmA, k0, m0, za, full_bar(stage));
            }
            if constexpr (B_MN) {
#pragma unroll
              for (int h = 0; h < C_::B_COLS / 64; ++h)
                tma_load_3d(sb + (uint32_t)h * 8192u, &tmB, n0 + 64 * h, k0, zb, full_bar(stage));
            } else {
              tma_load_3d(sb, &tmB, k0, n0, zb, full_bar(stage));
            }
            pending |= 1u << stage;
            pend_phase = (pend_phase & ~(1u << stage)) | (phase << stage);
          } else {
            pending &= ~(1u << stage);
          }
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      // Drain: every load issued must land before the block can exit.
      for (int s = 0; s < STAGES; ++s)
        if (pending & (1u << s)) mbar_wait_drain(full_bar(s), (pend_phase >> s) & 1u, p.timeout_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // 2-SM pairs: only the even block issues MMAs
    if (lane == 0 && (!TWO_SM || rank == 0)) {
      constexpr uint32_t idesc = make_idesc<BN, A_MN, B_MN, TWO_SM ? 2 * BM : BM, Elem<T>::FMT>();
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      Unit U;
      for (; ok && unit_at<PAIR, BN>(p, worker, workers, it, rank, U); ++it) {
        const int nkb = U.nkb;
        const int buf = it & 1;
        const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
        if (!mbar_wait(acce_bar(buf), acc_phase ^ 1u, wc)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * BN);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = tiles_addr + (uint32_t)(stage * C_::STAGE_BYTES);
          const uint32_t sb = sa + (uint32_t)A_TILE_BYTES;
#pragma unroll
          for (int kk = 0; kk < kblk<T>() / kmma<T>(); ++kk) {
            uint64_t ad, bd;
            if constexpr (A_MN) ad = make_sdesc(sa + (uint32_t)kk * 2048u, 8192u, 1024u);
            else ad = make_sdesc(sa + (uint32_t)kk * 32u, 16u, 1024u);
            if constexpr (B_MN) bd = make_sdesc(sb + (uint32_t)kk * 2048u, 8192u, 1024u);
            else bd = make_sdesc(sb + (uint32_t)kk * 32u, 16u, 1024u);
            const uint32_t acc = (kb | kk) != 0 ? 1u : 0u;
            if constexpr (sizeof(T) == 4) {
              if constexpr (TWO_SM) tc_mma_tf32_pair(d_tmem, ad, bd, idesc, acc);
              else tc_mma_tf32(d_tmem, ad, bd, idesc, acc);
            } else {
              if constexpr (TWO_SM) tc_mma_f16_pair(d_tmem, ad, bd, idesc, acc);
              else tc_mma_f16(d_tmem, ad, bd, idesc, acc);
            }
          }
          // buffer free once these MMAs finish (in both blocks of a pair)
          if constexpr (TWO_SM) tc_commit_pair_mc(empty_bar(stage), (uint16_t)3u);
          else tc_commit(empty_bar(stage));
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        // accumulator complete (2-SM pairs: in both blocks' tensor memory)
        if constexpr (TWO_SM) tc_commit_pair_mc(accf_bar(buf), (uint16_t)3u);
        else tc_commit(accf_bar(buf));
      }
      // Drain: every MMA issued must finish before tensor memory is freed.
      if constexpr (TWO_SM) tc_commit_pair_mc(drain_bar, (uint16_t)1u);
      else tc_commit(drain_bar);
      mbar_wait_drain(drain_bar, 0u, p.timeout_ns);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // this warp may access TMEM lanes 32q .. 32q+31
    const int row = q * 32 + lane;
    const int ew = warp - 2;                 // epilogue warp index, 0 .. EPI_WARPS-1
    const int hh = ew / 4;                   // which share of the columns it drains
    const int nh = p.epi_halves;             // shares in use (long-K tiles use one)
    // this warp's 32-column chunks [c_lo, c_hi) and 64-column groups [g_lo, g_hi)
    const int c_lo = (BN / 32) * hh / nh, c_hi = (BN / 32) * (hh + 1) / nh;
    const int g_lo = (BN / 64) * hh / nh, g_hi = (BN / 64) * (hh + 1) / nh;
    // staging buffers of this warp (the block's 4 KiB buffers split over the
    // warps in use)
    const int nbw = (C_::STAGING_BYTES / 4096) / (4 * nh);
    auto wait_staging = [&]() {  // this warp's oldest store has read its buffer
      if (lane == 0) {
        if (nbw >= 2) bulk_wait_read<1>();
        else bulk_wait_read<0>();
      }
      __syncwarp();
    };
    // the accumulator buffer is released by every epilogue thread once its
    // last tensor-memory load of the unit is done
    auto release_acc = [&](int buf) {
      tc_fence_before();
      if constexpr (TWO_SM) mbar_arrive_cluster(mapa_shared(acce_bar(buf), 0u));
      else mbar_arrive(acce_bar(buf));
    };
    // TMA stores: C boxes of 32 rows (64 columns of 16-bit C, 32 of fp32),
    // numbered i in [i_lo, i_hi) within a unit, take this warp's buffers in
    // turn across units (box i at buffer (nb0 + i - i_lo) % nbw, nb0 the
    // boxes of earlier units), so the buffer written next is always the
    // least recently stored from.  With beta != 0, C comes in by TMA loads of
    // the same boxes into the buffers, ahead of use; lane 0 alone tracks which
    // buffers have a load in flight (cpend) and their barriers' phases (cph).
    // (fp32 C with one buffer a warp: the load of each 32-column box would be
    // waited for in turn -- measured slower than the direct path, which keeps
    // eight 16-byte loads a thread in flight -- so that case takes the latter)
    constexpr int KBOX = 128 / (int)sizeof(T);
    const bool tma_c = p.c_tma && (p.beta == 0.f || sizeof(T) == 2 || nbw >= 2);
    const bool c_in = tma_c && p.beta != 0.f;
    const int i_lo = sizeof(T) == 4 ? c_lo : g_lo, i_hi = sizeof(T) == 4 ? c_hi : g_hi;
    // 32-column chunks of a shared tile this warp publishes, sums and
    // counts: the chunks its store of the tile will cover (64-column groups
    // for 16-bit C through TMA, 32-column chunks otherwise), so that a warp
    // only ever stores columns whose sums it finished itself
    const int s_lo = (sizeof(T) == 2 && tma_c) ? 2 * g_lo : c_lo;
    const int s_hi = (sizeof(T) == 2 && tma_c) ? 2 * g_hi : c_hi;
    int nb = 0;
    uint32_t cpend = 0u, cph = 0u;
    auto c_load = [&](int lb, int gx, int gy, int bz_) {  // lane 0
      const int bi = ew * nbw + lb;
      bulk_wait_read<0>();  // earlier stores from the buffer have read it
      mbar_arrive_expect_tx(cload_bar(bi), 4096u);
      tma_load_3d(staging_addr + (uint32_t)(bi * 4096), &tmC, gx, gy, bz_, cload_bar(bi));
      cpend |= 1u << lb;
    };
    auto c_wait = [&](int lb) -> bool {  // whole warp
      bool ok = true;
      if (lane == 0 && ((cpend >> lb) & 1u)) {
        ok = mbar_wait(cload_bar(ew * nbw + lb), (cph >> lb) & 1u, wc);
        if (ok) { cph ^= 1u << lb; cpend &= ~(1u << lb); }
      }
      return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    };
    int it = 0;
    bool dead = false;
    uint32_t fph = 0u;  // phase of this warp's fix_bar (lane 0)
    Unit U;
    // (warps of an unused share take no unit; they wait at the final barrier)
    for (; hh < nh && !dead && unit_at<PAIR, BN>(p, worker, workers, it, rank, U); ++it) {
      const int m0 = U.m0, n0 = U.n0, bz = U.bz;
      const int buf = it & 1;
      const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
      // C of the first boxes is requested ahead (a box wholly past M or N is
      // neither loaded nor stored): for a whole tile before its accumulator
      // is ready
      const bool c_rows = m0 + q * 32 < p.M;
      const int nb0 = nb;
      auto box_buf = [&](int i) { return (nb0 + i - i_lo) % nbw; };
      auto prefetch_c = [&]() {
        if (c_in && c_rows && lane == 0)
          for (int i = i_lo; i < i_hi && i < i_lo + nbw; ++i)
            if (n0 + KBOX * i < p.N) c_load(box_buf(i), n0 + KBOX * i, m0 + q * 32, bz);
      };
      if (U.sk < 0) prefetch_c();
      // Shared tile: its contributors (ranges w_first .. w_last, in K order),
      // this strip's arrival counter, and whether this is the worker's last
      // unit -- which reads the counter before its accumulator is ready, so
      // that the read's latency overlaps the main loop.
      int64_t s0 = 0;
      int w_first = 0, w_last = 0;
      unsigned int* cnt = nullptr;
      bool final = false;
      unsigned int seen = 0;
      if (U.sk >= 0) {
        s0 = (int64_t)U.sk * p.steps;
        w_first = sk_owner(p, s0);
        w_last = sk_owner(p, s0 + p.steps - 1);
        cnt = p.sk_cnt + (((int64_t)U.sk * (PAIR ? 2 : 1) + rank) * 4 + q) * EPI_HALVES + hh;
        Unit U2;
        final = !unit_at<PAIR, BN>(p, worker, workers, it + 1, rank, U2);
        if (!p.sk_publish && final && lane == 0 && s_lo < s_hi) seen = ld_acquire(cnt);
      }
      // one lane waits, the warp follows: the TMEM loads below are
      // warp-collective, so the whole warp must take the same branch
      bool got = false;
      if (lane == 0) got = mbar_wait(accf_bar(buf), acc_phase, wc);
      got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
      if (!got) break;
      tc_fence_after();
      const int gm = m0 + row;
      const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN);
      // shared tile: a warp's 32 x BN partial sums live in its strip of the
      // range's slot, laid out as the warp holds them -- [chunk c][float4 v]
      // [lane] -- so every store and load of a warp covers 512 contiguous
      // bytes
      constexpr int P = PAIR ? 2 : 1;
      constexpr int STRIP = 32 * BN;  // floats per warp strip
      auto strip_of = [&](int w_, int slot_) {
        return p.sk_ws + ((((int64_t)w_ * 2 + slot_) * P + rank) * 4 + q) * STRIP;
      };
      bool whole = U.sk < 0;
      if (!whole) {
        // ------------------------------------------------ shared tile
        // The contributor that finds every other one counted in, and is on
        // its last unit, adds their sums to its own accumulator (bulk copies
        // into the stage ring, idle once the worker's last accumulator is
        // complete) and stores the tile as a whole one.  Any other
        // contributor publishes its sums in its slot and counts in; if that
        // makes it the last, it finishes the strip the same way (on its last
        // unit) or from the slots with plain loads (earlier units, rare).
        if (s_lo == s_hi) { release_acc(buf); continue; }  // (no columns: not counted)
        const int n_contrib = w_last - w_first + 1;
        if (p.sk_publish) {
          // publish only: the reduction kernel finishes every shared tile
          float* const mine = strip_of(worker, U.slot);
#pragma unroll 1
          for (int c = s_lo; c < s_hi; ++c) {
            uint32_t r[32];
            __syncwarp();
            tmem_ld_32x32b_x32(t_row + (uint32_t)(c * 32), r);
            tmem_ld_wait();
            if (c == s_hi - 1) release_acc(buf);
            float4* dst = reinterpret_cast<float4*>(mine) + c * 256 + lane;
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[v * 32] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                        __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
          }
          continue;
        }
        constexpr uint32_t RING = (uint32_t)(STAGES * C_::STAGE_BYTES);
        const uint32_t region_bytes = (RING / (uint32_t)(4 * nh)) & ~4095u;
        const int n_slots = (int)(region_bytes >> 12);
        const uint32_t region = tiles_addr + (uint32_t)(hh * 4 + q) * region_bytes;
        seen = __shfl_sync(0xffffffffu, seen, 0);
        if (final && seen != (unsigned int)(n_contrib - 1)) {  // look again
          if (lane == 0) seen = ld_acquire(cnt);
          seen = __shfl_sync(0xffffffffu, seen, 0);
        }
        const bool ring_ok = n_contrib - 1 <= n_slots;
        if (!(final && ring_ok && seen == (unsigned int)(n_contrib - 1))) {
          // publish this range's sums in its slot, then count in
          float* const mine = strip_of(worker, U.slot);
#pragma unroll 1
          for (int c = s_lo; c < s_hi; ++c) {
            uint32_t r[32];
            __syncwarp();
            tmem_ld_32x32b_x32(t_row + (uint32_t)(c * 32), r);
            tmem_ld_wait();
            if (!final && c == s_hi - 1) release_acc(buf);
            float4* dst = reinterpret_cast<float4*>(mine) + c * 256 + lane;
#pragma unroll
            for (int v = 0; v < 8; ++v)
              dst[v * 32] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                        __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
          }
          __threadfence();
          __syncwarp();
          unsigned int old = 0;
          if (lane == 0) old = atomicAdd(cnt, 1u);
          old = __shfl_sync(0xffffffffu, old, 0);
          if (old != (unsigned int)(n_contrib - 1)) {  // another contributor finishes it
            if (final) release_acc(buf);
            continue;
          }
          __threadfence();  // every contributor's sums are visible
          if (!final || !ring_ok) {
            // every slot (this range's own included), plain loads, K order
#pragma unroll 1
            for (int c = s_lo; c < s_hi; ++c) {
              float v[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = 0.f;
              for (int w2 = w_first; w2 <= w_last; ++w2) {
                const float4* src =
                    reinterpret_cast<const float4*>(strip_of(w2, sk_slot(p, w2, s0))) + c * 256 + lane;
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                  const float4 f = __ldcg(src + w * 32);
                  v[4 * w] += f.x; v[4 * w + 1] += f.y; v[4 * w + 2] += f.z; v[4 * w + 3] += f.w;
                }
              }
              if (gm < p.M) store_c32<T>(p, bz, gm, n0 + c * 32, v);
            }
            if (final) release_acc(buf);
            __syncwarp();
            if (lane == 0) atomicExch(cnt, 0u);
            continue;
          }
        }
        // Add the other contributors' sums to this accumulator strip, in K
        // order, through this warp's share of the ring (4 KiB slots, one
        // 32-column chunk of one contributor each).
        {
          const int per = n_contrib - 1;
          const int cpb = n_slots / per > 0 ? n_slots / per : 1;
          bool ok = true;
          for (int c0 = s_lo; c0 < s_hi && ok; c0 += cpb) {
            const int c1 = min(s_hi, c0 + cpb);
            if (lane == 0) {
              fence_proxy_async_global();
              mbar_arrive_expect_tx(fix_bar(ew), (uint32_t)((c1 - c0) * per) * 4096u);
              int sl = 0;
              for (int c = c0; c < c1; ++c)
                for (int w2 = w_first; w2 <= w_last; ++w2) {
                  if (w2 == worker) continue;
                  bulk_load(region + (uint32_t)sl * 4096u,
                            strip_of(w2, sk_slot(p, w2, s0)) + c * 1024, 4096u, fix_bar(ew));
                  ++sl;
                }
              ok = mbar_wait(fix_bar(ew), fph, wc);
              // (given up: the copies in flight land before the block's
              // shared memory is released)
              if (!ok) mbar_wait_drain(fix_bar(ew), fph, p.timeout_ns);
              fph ^= 1u;
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
            int sl = 0;
#pragma unroll 1
            for (int c = c0; c < c1; ++c) {
              uint32_t r[32];
              __syncwarp();
              tmem_ld_32x32b_x32(t_row + (uint32_t)(c * 32), r);
              tmem_ld_wait();
              float v[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = 0.f;
              for (int w2 = w_first; w2 <= w_last; ++w2) {
                if (w2 == worker) {
#pragma unroll
                  for (int j = 0; j < 32; ++j) v[j] += __uint_as_float(r[j]);
                  continue;
                }
                const uint32_t a = region + (uint32_t)sl * 4096u + (uint32_t)lane * 16u;
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                  float f0, f1, f2, f3;
                  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                               : "=f"(f0), "=f"(f1), "=f"(f2), "=f"(f3)
                               : "r"(a + (uint32_t)w * 512u)
                               : "memory");
                  v[4 * w] += f0; v[4 * w + 1] += f1; v[4 * w + 2] += f2; v[4 * w + 3] += f3;
                }
                ++sl;
              }
#pragma unroll
              for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(v[j]);
              tmem_st_32x32b_x32(t_row + (uint32_t)(c * 32), r);
            }
            tmem_st_wait();
            __syncwarp();  // every lane has read the slots before they are refilled
          }
          if (!ok) { dead = true; break; }
        }
        if (lane == 0) atomicExch(cnt, 0u);
        whole = true;
        prefetch_c();
      }
      if constexpr (sizeof(T) == 4) if (whole && tma_c) {
        // fp32 C through TMA stores, 32 columns (128 bytes a row) at a time,
        // in the same 128-byte swizzle as the 16-bit path below
        // (two copies of the loop: with C loads (beta != 0) and without)
        auto boxes = [&](auto cin_tag) {
          constexpr bool CIN = decltype(cin_tag)::value;
          const bool epi = p.ep.bias != nullptr || p.ep.act != 0;
          if (c_lo == c_hi) release_acc(buf);
#pragma unroll 1
          for (int c = c_lo; c < c_hi; ++c) {
            // request C of box c + nbw - 1 into the buffer box c - 1 used
            if (CIN && c > c_lo && lane == 0 && c_rows && c + nbw - 1 < c_hi &&
                n0 + 32 * (c + nbw - 1) < p.N)
              c_load(box_buf(c + nbw - 1), n0 + 32 * (c + nbw - 1), m0 + q * 32, bz);
            uint32_t r[32];
            __syncwarp();
            tmem_ld_32x32b_x32(t_row + (uint32_t)(c * 32), r);
            tmem_ld_wait();
            if (c == c_hi - 1) release_acc(buf);
            const int gn0 = n0 + c * 32;
            const uint32_t sbuf = staging_addr + (uint32_t)((ew * nbw + box_buf(c)) * 4096);
            if (CIN) {
              if (!c_wait(box_buf(c))) { dead = true; break; }
            } else {
              wait_staging();
            }
#pragma unroll
            for (int w = 0; w < 8; ++w) {
              const uint32_t dst = sbuf + (uint32_t)(lane * 128 + ((w ^ (lane & 7)) * 16));
              float cv[4] = {0.f, 0.f, 0.f, 0.f};
              if (CIN)
                asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                             : "=f"(cv[0]), "=f"(cv[1]), "=f"(cv[2]), "=f"(cv[3])
                             : "r"(dst)
                             : "memory");
              float x[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                x[e] = p.alpha * __uint_as_float(r[4 * w + e]);
                if (CIN) x[e] = __fmaf_rn(p.beta, cv[e], x[e]);
                const int col = gn0 + 4 * w + e;
                if (epi && col < p.N) x[e] = apply_epilogue<T>(x[e], p.ep, col);
              }
              asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "f"(x[0]),
                           "f"(x[1]), "f"(x[2]), "f"(x[3])
                           : "memory");
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && c_rows && gn0 < p.N) {
              tma_store_3d(&tmC, gn0, m0 + q * 32, bz, sbuf);
              bulk_commit();
            }
          }
        };
        if (c_in) boxes(std::true_type{});
        else boxes(std::false_type{});
        nb += i_hi - i_lo;
        continue;
      }
      if constexpr (sizeof(T) == 2) if (whole && tma_c) {
        // C through TMA stores, 64 columns at a time: two tensor-memory loads
        // in flight, the 32 x 64 16-bit block packed into this warp's staging
        // buffer in the 128-byte swizzle (16-byte chunk w of row l at chunk
        // w ^ (l & 7): the 8 lanes of each store phase hit distinct banks),
        // then one TMA store clipped by the unit at M and N
        // (two copies of the loop: with C loads (beta != 0) and without)
        auto boxes = [&](auto cin_tag) {
          constexpr bool CIN = decltype(cin_tag)::value;
          const bool epi = p.ep.bias != nullptr || p.ep.act != 0;
          if (g_lo == g_hi) release_acc(buf);
#pragma unroll 1
          for (int g = g_lo; g < g_hi; ++g) {
            // request C of box g + nbw - 1 into the buffer box g - 1 used
            if (CIN && g > g_lo && lane == 0 && c_rows && g + nbw - 1 < g_hi &&
                n0 + 64 * (g + nbw - 1) < p.N)
              c_load(box_buf(g + nbw - 1), n0 + 64 * (g + nbw - 1), m0 + q * 32, bz);
            const int c = 2 * g;
            uint32_t r0[32], r1[32];
            __syncwarp();
            tmem_ld_32x32b_x32(t_row + (uint32_t)(c * 32), r0);
            tmem_ld_32x32b_x32(t_row + (uint32_t)(c * 32 + 32), r1);
            tmem_ld_wait();
            if (g == g_hi - 1) release_acc(buf);
            const int gn0 = n0 + c * 32;
            const uint32_t sbuf = staging_addr + (uint32_t)((ew * nbw + box_buf(g)) * 4096);
            if (CIN) {
              if (!c_wait(box_buf(g))) { dead = true; break; }
            } else {
              wait_staging();
            }
            // 16-byte chunk w (columns 8w .. 8w+7 of the 64) of this lane's row;
            // r holds columns 32h .. 32h+31 (constant indices after unrolling)
            auto pack_half = [&](const uint32_t (&r)[32], int h) {
#pragma unroll
              for (int ww = 0; ww < 4; ++ww) {
                const int w = 4 * h + ww;
                const uint32_t dst = sbuf + (uint32_t)(lane * 128 + ((w ^ (lane & 7)) * 16));
                uint4 ci = make_uint4(0u, 0u, 0u, 0u);
                if (CIN)
                  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                               : "=r"(ci.x), "=r"(ci.y), "=r"(ci.z), "=r"(ci.w)
                               : "r"(dst)
                               : "memory");
                const typename Elem<T>::T2* ch = reinterpret_cast<const typename Elem<T>::T2*>(&ci);
                uint4 o;
                typename Elem<T>::T2* oh = reinterpret_cast<typename Elem<T>::T2*>(&o);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  float x0 = p.alpha * __uint_as_float(r[8 * ww + 2 * e]);
                  float x1 = p.alpha * __uint_as_float(r[8 * ww + 2 * e + 1]);
                  if (CIN) {
                    const float2 cf = Elem<T>::unpack(ch[e]);
                    x0 = __fmaf_rn(p.beta, cf.x, x0);
                    x1 = __fmaf_rn(p.beta, cf.y, x1);
                  }
                  if (epi) {
                    // (columns past N are clipped by the store; their bias is not read)
                    const int col = gn0 + 8 * w + 2 * e;
                    if (col < p.N) x0 = apply_epilogue<T>(x0, p.ep, col);
                    if (col + 1 < p.N) x1 = apply_epilogue<T>(x1, p.ep, col + 1);
                  }
                  oh[e] = Elem<T>::pack(x0, x1);
                }
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(o.x),
                             "r"(o.y), "r"(o.z), "r"(o.w)
                             : "memory");
              }
            };
            pack_half(r0, 0);
            pack_half(r1, 1);
            fence_proxy_async_smem();
            __syncwarp();
            // (a block wholly past M or N -- the second tile of a pair on an odd
            // tile-row count -- is not stored at all)
            if (lane == 0 && c_rows && gn0 < p.N) {
              tma_store_3d(&tmC, gn0, m0 + q * 32, bz, sbuf);
              bulk_commit();
            }
          }
        };
        if (c_in) boxes(std::true_type{});
        else boxes(std::false_type{});
        nb += i_hi - i_lo;
        continue;
      }
      // (2-SM pairs: the even block's MMAs write both blocks' tensor memory,
      // so the release goes to its barrier)
      if (c_lo == c_hi) release_acc(buf);
#pragma unroll 1
      for (int c = c_lo; c < c_hi; ++c) {
        uint32_t r[32];
        __syncwarp();
        tmem_ld_32x32b_x32(t_row + (uint32_t)(c * 32), r);
        tmem_ld_wait();
        if (c == c_hi - 1) release_acc(buf);
        const int gn0 = n0 + c * 32;
        if (!p.c_vec_ok) {
          // through this warp's first staging buffer (no TMA store uses the
          // buffers in a launch that takes this path); the whole warp takes
          // part, rows past M are skipped inside
          if (m0 + q * 32 < p.M)
            store_c32_staged<T>(p, bz, m0 + q * 32, gn0,
                                staging_addr + (uint32_t)(ew * nbw * 4096), r, lane);
          continue;
        }
        // rows past M: loaded (warp-collective) but not stored
        if (gm >= p.M) continue;
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
        store_c32<T>(p, bz, gm, gn0, v);
      }
    }
    if (lane == 0) {
      bulk_wait_all();  // C stores complete before the block ends
      // (after an abort: C loads still in flight land before shared memory
      // is released)
      for (int lb = 0; lb < nbw; ++lb)
        if ((cpend >> lb) & 1u)
          mbar_wait_drain(cload_bar(ew * nbw + lb), (cph >> lb) & 1u, p.timeout_ns);
    }
  }

  tc_fence_before();
  // A pair leaves together: the peer's copies and commit arrivals target
  // this block's shared memory until both are done.
  if constexpr (PAIR) cluster_sync();
  else __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    if constexpr (TWO_SM) tmem_dealloc_pair(tmem_base, (uint32_t)C_::TMEM_COLS);
    else tmem_dealloc(tmem_base, (uint32_t)C_::TMEM_COLS);
  }
}

// Reduction of shared tiles published by every contributor (sk_publish):
// one block of 256 threads per (shared tile, block of the pair, 32-row
// quarter, 32-column chunk).  Thread (v, lane) loads float4 v of row lane
// from every contributor (all loads in flight together; every load of a warp
// covers 512 contiguous bytes) and adds them in K order; the 32 x 32 sums go
// through shared memory so that the output is written 4 columns a thread,
// 8 threads a row -- 64-byte (16-bit C) or 128-byte (fp32 C) row segments --
// as act(alpha * sum + beta * C + bias).  Launched after the GEMM kernel in
// stream order.
template <typename T, bool PAIR, int TBN>
__global__ void __launch_bounds__(256) hgemm_sk_reduce(const HParams p) {
  using E = Elem<T>;
  pdl_wait();
  pdl_trigger();
  constexpr int P = PAIR ? 2 : 1;
  constexpr int CH = TBN / 32;
  constexpr int STRIP = 32 * TBN;
  // contributors a tile can have: the planner allows at most 5 to tiles wider
  // than 64 columns, 16 to narrower ones
  constexpr int MAXC = TBN > 64 ? 5 : 16;
  __shared__ float sum[32][33];
  const int lane = threadIdx.x & 31, v = threadIdx.x >> 5;
  const int64_t unit = blockIdx.x;
  const int c = (int)(unit % CH);
  const int q = (int)((unit / CH) % 4);
  const int rank = (int)((unit / (CH * 4)) % P);
  const int64_t tr = unit / (CH * 4 * P);
  if (tr >= (int64_t)p.tiles - p.dp_tiles) return;
  int m0, n0, bz;
  tile_origin<PAIR, TBN>(p, p.dp_tiles + (int)tr, rank, m0, n0, bz);
  const int64_t s0 = tr * p.steps;
  const int w_first = sk_owner(p, s0), w_last = sk_owner(p, s0 + p.steps - 1);
  if (w_first == w_last) return;  // one range covered the tile: stored as a whole one
  // (only the first contributor can have started before the tile: slot 1)
  const int slot0 = sk_slot(p, w_first, s0);
  float4 f[MAXC];
#pragma unroll
  for (int i = 0; i < MAXC; ++i) {
    const int w2 = w_first + i;
    f[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (w2 <= w_last)
      f[i] = __ldcg(reinterpret_cast<const float4*>(
                        p.sk_ws + ((((int64_t)w2 * 2 + (i == 0 ? slot0 : 0)) * P + rank) * 4 + q) *
                                      STRIP) +
                    c * 256 + v * 32 + lane);
  }
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
  for (int i = 0; i < MAXC; ++i) {
    if (w_first + i > w_last) break;
    a0 += f[i].x; a1 += f[i].y; a2 += f[i].z; a3 += f[i].w;
  }
  sum[lane][4 * v] = a0; sum[lane][4 * v + 1] = a1;
  sum[lane][4 * v + 2] = a2; sum[lane][4 * v + 3] = a3;
  __syncthreads();
  // thread t: row t / 8 of the chunk, columns 4 (t % 8) .. +3
  const int r = threadIdx.x >> 3, cc = (threadIdx.x & 7) * 4;
  const int gm = m0 + q * 32 + r, gn0 = n0 + c * 32 + cc;
  if (gm >= p.M || gn0 >= p.N) return;
  T* dst = static_cast<T*>(p.C) + (int64_t)bz * p.stride_c + (int64_t)gm * p.ldc + gn0;
  const bool epi = p.ep.bias != nullptr || p.ep.act != 0;
  float x[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) x[j] = p.alpha * sum[r][cc + j];
  // 16 (fp32) or 8 (16-bit) aligned bytes when C rows are 16-byte aligned
  const bool vec = p.c_vec_ok && gn0 + 3 < p.N;
  if (p.beta != 0.f) {
    if (vec && sizeof(T) == 4) {
      const float4 cv = *reinterpret_cast<const float4*>(dst);
      x[0] = __fmaf_rn(p.beta, cv.x, x[0]); x[1] = __fmaf_rn(p.beta, cv.y, x[1]);
      x[2] = __fmaf_rn(p.beta, cv.z, x[2]); x[3] = __fmaf_rn(p.beta, cv.w, x[3]);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (gn0 + j < p.N) x[j] = __fmaf_rn(p.beta, E::to(dst[j]), x[j]);
    }
  }
  if (epi) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (gn0 + j < p.N) x[j] = apply_epilogue<T>(x[j], p.ep, gn0 + j);
  }
  if (vec) {
    if constexpr (sizeof(T) == 4) {
      *reinterpret_cast<float4*>(dst) = make_float4(x[0], x[1], x[2], x[3]);
    } else {
      typename E::T2 h[2] = {E::pack(x[0], x[1]), E::pack(x[2], x[3])};
      *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(h);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (gn0 + j < p.N) dst[j] = E::from(x[j]);
  }
}

// ---------------------------------------------------------------- host side
// How many two-block clusters of the pair kernel can be resident at once
// (fewer than SMs / 2 when the SMs of a GPC do not all pair up).  Queried once
// per kernel configuration.
template <typename T, int BN, bool A_MN, bool B_MN, int MODE>
int pair_slots(int num_sms) {
  static int n = 0;
  if (n == 0) {
    using C_ = Cfg<BN, B_MN, MODE>;
    auto kern = hgemm_tc_kernel<T, BN, A_MN, B_MN, MODE>;
    int q = 0;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C_::SMEM_BYTES) == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(2 * (num_sms / 2));
      cfg.blockDim = dim3(THREADS);
      cfg.dynamicSmemBytes = C_::SMEM_BYTES;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&q, kern, &cfg) != cudaSuccess) q = 0;
    }
    n = q > 0 ? q : num_sms / 2;
  }
  return n;
}

// cudaFuncSetAttribute for the kernel's shared memory, once per
// configuration (a driver call per GEMM otherwise).
template <typename T, int BN, bool A_MN, bool B_MN, int MODE>
cudaError_t kernel_attributes() {
  static const cudaError_t e = cudaFuncSetAttribute(
      hgemm_tc_kernel<T, BN, A_MN, B_MN, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
      Cfg<BN, B_MN, MODE>::SMEM_BYTES);
  return e;
}

template <typename T, int BN, bool A_MN, bool B_MN, int MODE>
cudaError_t launch_cfg(const HgemmArgs& a, const HParams& p, LaunchCtx& ctx) {
  constexpr CUtensorMapDataType TY = Elem<T>::TMA;
  constexpr bool PAIR = MODE != 0;
  using C_ = Cfg<BN, B_MN, MODE>;
  CUtensorMap mA, mB;
  bool ok;
  const CUtensorMapSwizzle SW = CU_TENSOR_MAP_SWIZZLE_128B;
  // a pitch-0 operand is one matrix shared by every batch entry (z stays 0);
  // 3xTF32 operands are two planes each (hi, lo)
  const int64_t nba = a.split3 ? 2 : (p.za_mask ? a.batch : 1);
  const int64_t nbb = a.split3 ? 2 : (p.zb_mask ? a.batch : 1);
  // K-major boxes are one 128-byte swizzle row deep in K (64 16-bit or 32
  // fp32 elements); MN-major boxes (16-bit types only) are 64 x 64
  constexpr int KB = kblk<T>(), ES = (int)sizeof(T);
  if (A_MN) ok = make_map(&mA, TY, a.A, a.K, a.M, a.lda, 64, 64, SW, nba, a.stride_a, ES);  // [K, M]
  else ok = make_map(&mA, TY, a.A, a.M, a.K, a.lda, KB, BM, SW, nba, a.stride_a, ES);       // [M, K]
  if (!ok) return cudaErrorNotSupported;
  if (B_MN) ok = make_map(&mB, TY, a.B, a.K, a.N, a.ldb, 64, 64, SW, nbb, a.stride_b, ES);  // [K, N]
  else ok = make_map(&mB, TY, a.B, a.N, a.K, a.ldb, KB, PAIR ? BN / 2 : BN, SW, nbb,
                     a.stride_b, ES);                                                          // [N, K]
  if (!ok) return cudaErrorNotSupported;
  // C: row-major [M, N], 128-byte x 32-row boxes (64 x 32 16-bit, 32 x 32 fp32),
  // 128-byte swizzle (used only when p.c_tma)
  CUtensorMap mC;
  memset(&mC, 0, sizeof(mC));
  if (p.c_tma && !make_map(&mC, TY, a.C, a.M, a.N, a.ldc, KB, 32, CU_TENSOR_MAP_SWIZZLE_128B,
                           p.batch, p.stride_c, ES))
    return cudaErrorNotSupported;
  auto kern = hgemm_tc_kernel<T, BN, A_MN, B_MN, MODE>;
  cudaError_t e = kernel_attributes<T, BN, A_MN, B_MN, MODE>();
  if (e != cudaSuccess) return e;
  // both epilogue shares only where this configuration's staging has room
  HParams pp = p;
  if (!C_::EPI2) pp.epi_halves = 1;
  const int workers = a.plan.workers;
  ctx.grid = PAIR ? 2 * workers : workers;
  e = launch_kernel(kern, dim3(ctx.grid), dim3(THREADS), C_::SMEM_BYTES, ctx.stream, PAIR ? 2 : 1,
                    mA, mB, mC, pp);
  if (e != cudaSuccess) return e;
  ctx.launches++;
  if (pp.sk_workers > 0 && pp.sk_publish) {
    const int64_t units = ((int64_t)pp.tiles - pp.dp_tiles) * (PAIR ? 2 : 1) * 4 * (BN / 32);
    e = launch_kernel(hgemm_sk_reduce<T, PAIR, BN>, dim3((unsigned)units), dim3(256), 0,
                      ctx.stream, 1, pp);
    if (e == cudaSuccess) ctx.launches++;
  }
  return e;
}

template <typename T, int BN>
cudaError_t launch_bn(const HgemmArgs& a, const HParams& p, LaunchCtx& ctx) {
  const bool A_MN = a.transA != 0, B_MN = a.transB == 0;
  constexpr bool CAN_PAIR = BN == 128 || BN == 256;
  constexpr int M2 = CAN_PAIR ? 2 : 0;
  const bool pair = CAN_PAIR && p.pair == 2;
  if constexpr (sizeof(T) == 4) {
    // TF32 operands are staged K-major only (the dispatcher packs them so)
    if (A_MN || B_MN) return cudaErrorInvalidValue;
    if (pair) return launch_cfg<T, BN, false, false, M2>(a, p, ctx);
    return launch_cfg<T, BN, false, false, 0>(a, p, ctx);
  } else {
#define GB300_HG(AM, BMN)                                                   \
  if (A_MN == AM && B_MN == BMN) {                                          \
    if (pair) return launch_cfg<T, BN, AM, BMN, M2>(a, p, ctx);             \
    return launch_cfg<T, BN, AM, BMN, 0>(a, p, ctx);                        \
  }
  GB300_HG(false, true)
  GB300_HG(true, true)
  GB300_HG(false, false)
  GB300_HG(true, false)
#undef GB300_HG
  }
  return cudaErrorInvalidValue;
}

// One launch of the kernel for element type T, as planned by hgemm_plan
// (tile width, pairs, schedule, scratch for shared tiles).
template <typename T>
cudaError_t launch_hgemm_t(const HgemmArgs& a, LaunchCtx& ctx) {
  const HPlan& pl = a.plan;
  HParams p;
  p.C = a.C;
  p.ldc = a.ldc;
  p.M = a.M; p.N = a.N; p.K = a.K;
  const int bn = a.bn;
  p.tiles_m = (a.M + BM - 1) / BM;
  p.tiles_n = (a.N + bn - 1) / bn;
  p.tiles = pl.tiles;
  p.steps = pl.steps;
  p.dp_tiles = pl.dp_tiles;
  p.sk_workers = pl.sk_workers;
  p.sk_steps = pl.sk_steps;
  auto magic = [](uint64_t d) { return d > 0 ? ~0ull / d : 0ull; };
  p.m_skw = magic((uint64_t)pl.sk_workers);
  p.m_sks = magic((uint64_t)pl.sk_steps);
  p.m_steps = magic((uint64_t)pl.steps);
  p.sk_ws = a.sk_ws;
  p.sk_cnt = a.sk_cnt;
  p.sk_publish = pl.sk_publish;
  p.alpha = a.alpha; p.beta = a.beta;
  p.status = ctx.status;
  p.timeout_ns = ctx.timeout_ns;
  p.fault_injection = a.fault_injection;
  constexpr int VEC = 16 / (int)sizeof(T);  // elements per 16 bytes
  p.c_vec_ok = ((reinterpret_cast<uintptr_t>(a.C) & 15u) == 0 && (a.ldc % VEC) == 0 &&
                (a.batch <= 1 || (a.stride_c % VEC) == 0)) ? 1 : 0;
  p.c_tma = (p.c_vec_ok && a.c_tma && bn >= (sizeof(T) == 4 ? 32 : 64)) ? 1 : 0;
  p.pair = pl.pair;
  p.batch = a.batch > 1 ? a.batch : 1;
  p.stride_c = p.batch > 1 ? a.stride_c : 0;
  p.za_mask = (p.batch > 1 && a.stride_a != 0) ? -1 : 0;
  p.zb_mask = (p.batch > 1 && a.stride_b != 0) ? -1 : 0;
  p.ep = a.ep;
  p.epi_halves = pl.epi_halves;
  p.split3 = a.split3;
  p.steps_k = a.split3 ? (a.K + kblk<T>() - 1) / kblk<T>() : 0;
  if (a.split3 && (sizeof(T) != 4 || p.batch > 1 || pl.steps != 3 * p.steps_k))
    return cudaErrorInvalidValue;
  if (pl.workers <= 0 || pl.steps <= 0 || pl.bn != bn) return cudaErrorInvalidValue;
  if (pl.sk_workers > 0 && (!a.sk_ws || (!pl.sk_publish && !a.sk_cnt))) return cudaErrorInvalidValue;
  switch (bn) {
    case 32: return launch_bn<T, 32>(a, p, ctx);
    case 64: return launch_bn<T, 64>(a, p, ctx);
    case 128: return launch_bn<T, 128>(a, p, ctx);
    case 192: return launch_bn<T, 192>(a, p, ctx);
    case 256: return launch_bn<T, 256>(a, p, ctx);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace
}  // namespace gb300
