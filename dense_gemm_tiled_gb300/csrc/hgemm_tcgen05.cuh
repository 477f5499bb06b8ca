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
//    (round to nearest even) -> global; or raw fp32 partial sums (split-K).
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
  static constexpr int FIXED_BYTES = 1024 /*align*/ + 256 /*barriers*/;
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
      STAGES * STAGE_BYTES + STAGING_BYTES + 1024 /*align*/ + 256 /*barriers*/;
};

struct HParams {
  void* C;  // __half or __nv_bfloat16, per the kernel's element type
  float* partial;
  int64_t ldc;
  int M, N, K;
  int k_slice;
  int tiles_m, tiles_n, splits;
  float alpha, beta;
  unsigned int* status;
  uint64_t timeout_ns;
  int fault_injection;
  int c_vec_ok;  // C base 16-byte aligned and ldc % 8 == 0
  int c_tma;     // C aligned: C leaves through TMA stores (and comes in by TMA loads)
  int pair;      // 2: clusters of two blocks run 2-SM (cta_group::2) MMAs; 0: single blocks
  // Tail split (only when splits == 1): units [0, dp_units) are whole tiles;
  // the remaining tiles are cut into tail_splits K slices of tail_k_slice, each
  // writing fp32 partials to tail_ws; per 32-row strip the last slice to
  // arrive (tail_cnt) sums all slices in slice order and runs the epilogue.
  int dp_units, tail_splits, tail_k_slice;
  // strided batch: units run over batch x tiles (no K split, no tail split);
  // the tensor maps carry the batch as their third coordinate
  int batch;
  int64_t stride_c;  // elements between consecutive C matrices
  int za_mask, zb_mask;  // -1: operand batched; 0: one matrix shared by all (pitch 0)
  Epilogue ep;           // bias (output type, per column) and activation
  int epi_halves;        // epilogue warps in use per accumulator quarter: 1 or EPI_HALVES
  float* tail_ws;          // [tail tiles][pair ? 2 : 1][tail_splits][4 warps][32 x BN]
  unsigned int* tail_cnt;  // [tail tiles][pair ? 2 : 1][4], zero on entry and on exit
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

// Work unit u -> tile, K range, slice.  Without pairs a tile is 128 x BN;
// with pairs (a cluster of two blocks sharing B) a unit covers two vertically
// adjacent tiles and block `rank` of the pair takes tile row 2 * pair_row + rank.
//  * split-K launches: unit = slice z of tile t, u = z * tiles + t;
//  * tail split: units below dp_units are whole tiles; unit dp_units + v is
//    slice v / tail_tiles of tail tile v % tail_tiles (`tail` >= 0);
//  * otherwise: unit = whole tile.
template <bool PAIR, int KB = BK>
__device__ __forceinline__ void unit_coords(int u, const HParams& p, int rank, int& m0, int& tn,
                                            int& kbeg, int& nkb, int& z, int& tail, int& bz) {
  const int rows = PAIR ? (p.tiles_m + 1) / 2 : p.tiles_m;
  const int tiles = rows * p.tiles_n;
  int t, ks;
  tail = -1;
  if (p.tail_splits > 0 && u >= p.dp_units) {
    const int tail_tiles = tiles - p.dp_units;
    const int v = u - p.dp_units;
    tail = v % tail_tiles;
    z = v / tail_tiles;
    t = p.dp_units + tail;
    ks = p.tail_k_slice;
  } else {
    z = u / tiles;
    t = u - z * tiles;
    ks = p.k_slice;
  }
  // a batched launch has no K split: the outer index is the batch entry
  bz = 0;
  if (p.batch > 1) {
    bz = z;
    z = 0;
  }
  const int per_group = GROUP_M * p.tiles_n;
  const int first_m = (t / per_group) * GROUP_M;
  const int gsize = min(rows - first_m, GROUP_M);
  const int tr = first_m + (t % per_group) % gsize;
  tn = (t % per_group) / gsize;
  const int tm = PAIR ? 2 * tr + rank : tr;
  m0 = tm * BM;
  kbeg = z * ks;
  const int kend = min(p.K, kbeg + ks);
  nkb = (kend - kbeg + KB - 1) / KB;
}

__device__ __forceinline__ int total_units(const HParams& p, bool pair) {
  const int tiles = (pair ? (p.tiles_m + 1) / 2 : p.tiles_m) * p.tiles_n;
  if (p.tail_splits > 0) return p.dp_units + (tiles - p.dp_units) * p.tail_splits;
  return tiles * p.splits * (p.batch > 1 ? p.batch : 1);
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

template <typename T, int BN, bool A_MN, bool B_MN, bool SPLIT, int MODE>
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
  static_assert(8 * (2 * STAGES + 6 + NSTAGING) <= 256, "barrier area");
  auto cload_bar = [&](int b) { return bar0 + 8u * (uint32_t)(2 * STAGES + 6 + b); };
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
  const int n_units = total_units(p, PAIR);

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
      for (int u = worker; u < n_units && ok; u += workers) {
        int m0, tn, kbeg, nkb, z, tail, bz;
        unit_coords<PAIR, kblk<T>()>(u, p, rank, m0, tn, kbeg, nkb, z, tail, bz);
        const int za = bz & p.za_mask, zb = bz & p.zb_mask;
        const int n0 = tn * BN;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, wc)) { ok = false; break; }
          const int k0 = kbeg + kb * kblk<T>();
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
      for (int u = worker; u < n_units && ok; u += workers, ++it) {
        int m0, tn, kbeg, nkb, z, tail, bz;
        unit_coords<PAIR, kblk<T>()>(u, p, rank, m0, tn, kbeg, nkb, z, tail, bz);
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
    const bool c_in = !SPLIT && tma_c && p.beta != 0.f;
    const int i_lo = sizeof(T) == 4 ? c_lo : g_lo, i_hi = sizeof(T) == 4 ? c_hi : g_hi;
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
    // (warps of an unused share take no unit; they wait at the final barrier)
    for (int u = hh < nh ? worker : n_units; u < n_units && !dead; u += workers, ++it) {
      int m0, tn, kbeg, nkb, z, tail, bz;
      unit_coords<PAIR, kblk<T>()>(u, p, rank, m0, tn, kbeg, nkb, z, tail, bz);
      const int n0 = tn * BN;
      const int buf = it & 1;
      const uint32_t acc_phase = (uint32_t)(it >> 1) & 1u;
      // C of the first boxes is requested before the accumulator is ready (a
      // box wholly past M or N is neither loaded nor stored)
      const bool c_rows = m0 + q * 32 < p.M;
      const int nb0 = nb;
      auto box_buf = [&](int i) { return (nb0 + i - i_lo) % nbw; };
      if (c_in && tail < 0 && c_rows && lane == 0)
        for (int i = i_lo; i < i_hi && i < i_lo + nbw; ++i)
          if (n0 + KBOX * i < p.N) c_load(box_buf(i), n0 + KBOX * i, m0 + q * 32, bz);
      // one lane waits, the warp follows: the TMEM loads below are
      // warp-collective, so the whole warp must take the same branch
      bool got = false;
      if (lane == 0) got = mbar_wait(accf_bar(buf), acc_phase, wc);
      got = __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
      if (!got) break;
      tc_fence_after();
      const int gm = m0 + row;
      const uint32_t t_row = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN);
      // tail slice: this warp's 32 x BN partial sums for the tile live in a
      // block of the workspace laid out as the warp holds them -- [chunk c]
      // [float4 v][lane] -- so every store and load of a warp covers 512
      // contiguous bytes
      constexpr int P = PAIR ? 2 : 1;
      constexpr int STRIP = 32 * BN;  // floats per warp strip
      float* const tail_strip =
          tail >= 0 ? p.tail_ws + ((((int64_t)(tail * P + rank) * p.tail_splits + z) * 4 + q) * STRIP)
                    : nullptr;
      if constexpr (sizeof(T) == 4) if (!SPLIT && tail < 0 && tma_c) {
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
      if constexpr (sizeof(T) == 2) if (!SPLIT && tail < 0 && tma_c) {
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
        if (tail >= 0) {
          float4* dst = reinterpret_cast<float4*>(tail_strip) + (c * 8) * 32 + lane;
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[v * 32] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                      __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
          continue;
        }
        const int gn0 = n0 + c * 32;
        if (!SPLIT && !p.c_vec_ok) {
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
        if constexpr (SPLIT) {
          float* dst = p.partial + ((int64_t)z * p.M + gm) * p.N + gn0;
          if (gn0 + 31 < p.N && (p.N & 3) == 0) {
#pragma unroll
            for (int v = 0; v < 8; ++v)
              reinterpret_cast<float4*>(dst)[v] =
                  make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                              __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
          } else {
            for (int j = 0; j < 32; ++j)
              if (gn0 + j < p.N) dst[j] = __uint_as_float(r[j]);
          }
        } else {
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
          store_c32<T>(p, bz, gm, gn0, v);
        }
      }
      if (tail >= 0 && c_lo < c_hi) {
        // Last slice to arrive for this 32-row strip (and column share)
        // finishes it: partial
        // writes are fenced before the arrival, the slices are summed in slice
        // order (so the result does not depend on which slice came last), and
        // the counter is left at zero for the next launch.  No waiting on
        // other blocks is involved.
        __threadfence();
        unsigned int old = 0;
        // one counter per 32-row strip and column share
        unsigned int* cnt = p.tail_cnt + ((tail * P + rank) * 4 + q) * EPI_HALVES + hh;
        if (lane == 0) old = atomicAdd(cnt, 1u);
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old == (unsigned int)(p.tail_splits - 1)) {
          __threadfence();
          const float* strip0 =
              p.tail_ws + (((int64_t)(tail * P + rank) * p.tail_splits * 4 + q) * STRIP);
          const int64_t slice_stride = 4 * (int64_t)STRIP;
#pragma unroll 1
          for (int c = c_lo; c < c_hi; ++c) {
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0.f;
            for (int zz = 0; zz < p.tail_splits; ++zz) {
              const float4* src =
                  reinterpret_cast<const float4*>(strip0 + zz * slice_stride) + (c * 8) * 32 + lane;
#pragma unroll
              for (int w = 0; w < 8; ++w) {
                const float4 f = __ldcg(src + w * 32);
                v[4 * w] += f.x; v[4 * w + 1] += f.y; v[4 * w + 2] += f.z; v[4 * w + 3] += f.w;
              }
            }
            if (gm < p.M) store_c32<T>(p, bz, gm, n0 + c * 32, v);
          }
          if (lane == 0) atomicExch(cnt, 0u);
        }
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

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 3-D tensor map over `batch` row-major [rows, cols] matrices of `esize`-byte
// elements with row pitch `ld` and batch pitch `stride` elements; box = box_cols (inner) x
// box_rows x 1, 128-byte swizzle by default, out-of-range elements read as
// zero.  Returns false when the driver rejects the description (the launch
// then reports cudaErrorNotSupported and nothing runs).
bool make_map(CUtensorMap* map, CUtensorMapDataType type, const void* base, int64_t rows,
              int64_t cols, int64_t ld, int box_cols, int box_rows,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B, int64_t batch = 1,
              int64_t stride = 0, int esize = 2) {
  auto enc = get_encode();
  if (!enc) return false;
  // [batch][rows][cols]; a single matrix is batch 1 with a nominal pitch
  if (batch <= 1) stride = ld * (rows > 0 ? rows : 1);
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)(batch > 1 ? batch : 1)};
  cuuint64_t strides[2] = {(cuuint64_t)(ld * esize), (cuuint64_t)(stride * esize)};
  cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, type, 3, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// How many two-block clusters of the pair kernel can be resident at once
// (fewer than SMs / 2 when the SMs of a GPC do not all pair up).  Queried once
// per kernel configuration.
template <typename T, int BN, bool A_MN, bool B_MN, int MODE>
int pair_slots(int num_sms) {
  static int n = 0;
  if (n == 0) {
    using C_ = Cfg<BN, B_MN, MODE>;
    auto kern = hgemm_tc_kernel<T, BN, A_MN, B_MN, false, MODE>;
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

int host_total_units(const HParams& p, bool pair) {
  const int tiles = (pair ? (p.tiles_m + 1) / 2 : p.tiles_m) * p.tiles_n;
  if (p.tail_splits > 0) return p.dp_units + (tiles - p.dp_units) * p.tail_splits;
  return tiles * p.splits * (p.batch > 1 ? p.batch : 1);
}

template <typename T, int BN, bool A_MN, bool B_MN, bool SPLIT, int MODE>
cudaError_t launch_cfg(const HgemmArgs& a, const HParams& p, LaunchCtx& ctx) {
  constexpr CUtensorMapDataType TY = Elem<T>::TMA;
  constexpr bool PAIR = MODE != 0;
  using C_ = Cfg<BN, B_MN, MODE>;
  CUtensorMap mA, mB;
  bool ok;
  const CUtensorMapSwizzle SW = CU_TENSOR_MAP_SWIZZLE_128B;
  // a pitch-0 operand is one matrix shared by every batch entry (z stays 0)
  const int64_t nba = p.za_mask ? a.batch : 1, nbb = p.zb_mask ? a.batch : 1;
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
  auto kern = hgemm_tc_kernel<T, BN, A_MN, B_MN, SPLIT, MODE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C_::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  // both epilogue shares only where this configuration's staging has room
  HParams pp = p;
  if (!C_::EPI2) pp.epi_halves = 1;
  if constexpr (PAIR) {
    // persistent grid of as many pairs as can be resident at once
    const int max_pairs = pair_slots<T, BN, A_MN, B_MN, MODE>(a.num_sms);
    const int units = host_total_units(p, true);
    const int pairs = units < max_pairs ? units : max_pairs;
    ctx.grid = 2 * pairs;
    e = launch_kernel(kern, dim3(2 * pairs), dim3(THREADS), C_::SMEM_BYTES, ctx.stream, 2, mA, mB,
                      mC, pp);
  } else {
    const int units = host_total_units(p, false);
    const int grid = units < a.num_sms ? units : a.num_sms;
    ctx.grid = grid;
    e = launch_kernel(kern, dim3(grid), dim3(THREADS), C_::SMEM_BYTES, ctx.stream, 1, mA, mB, mC,
                      pp);
  }
  if (e == cudaSuccess) ctx.launches++;
  return e;
}

template <typename T, int BN>
cudaError_t launch_bn(const HgemmArgs& a, const HParams& p, LaunchCtx& ctx) {
  const bool A_MN = a.transA != 0, B_MN = a.transB == 0, split = a.splits > 1;
  constexpr bool CAN_PAIR = BN == 128 || BN == 256;
  constexpr int M2 = CAN_PAIR ? 2 : 0;
  if constexpr (sizeof(T) == 4) {
    // TF32 operands are staged K-major only (the dispatcher packs them so)
    if (A_MN || B_MN) return cudaErrorInvalidValue;
    if (split) return launch_cfg<T, BN, false, false, true, 0>(a, p, ctx);
    if (CAN_PAIR && p.pair == 2) return launch_cfg<T, BN, false, false, false, M2>(a, p, ctx);
    return launch_cfg<T, BN, false, false, false, 0>(a, p, ctx);
  } else {
#define GB300_HG(AM, BMN)                                                   \
  if (A_MN == AM && B_MN == BMN) {                                          \
    if (split) return launch_cfg<T, BN, AM, BMN, true, 0>(a, p, ctx);       \
    if (CAN_PAIR && p.pair == 2) return launch_cfg<T, BN, AM, BMN, false, M2>(a, p, ctx); \
    return launch_cfg<T, BN, AM, BMN, false, 0>(a, p, ctx);                 \
  }
  GB300_HG(false, true)
  GB300_HG(true, true)
  GB300_HG(false, false)
  GB300_HG(true, false)
#undef GB300_HG
  }
  return cudaErrorInvalidValue;
}

// One launch of the kernel for element type T (HgemmArgs already planned by the
// dispatcher: tile width, split, pairs, tail).
template <typename T>
cudaError_t launch_hgemm_t(const HgemmArgs& a, LaunchCtx& ctx) {
  HParams p;
  p.C = a.C;
  p.partial = a.partial;
  p.ldc = a.ldc;
  p.M = a.M; p.N = a.N; p.K = a.K;
  p.splits = a.splits > 1 ? a.splits : 1;
  p.k_slice = a.splits > 1 ? a.k_slice : ((a.K + kblk<T>() - 1) / kblk<T>()) * kblk<T>();
  const int bn = a.bn;
  p.tiles_m = (a.M + BM - 1) / BM;
  p.tiles_n = (a.N + bn - 1) / bn;
  p.alpha = a.alpha; p.beta = a.beta;
  p.status = ctx.status;
  p.timeout_ns = ctx.timeout_ns;
  p.fault_injection = a.fault_injection;
  constexpr int VEC = 16 / (int)sizeof(T);  // elements per 16 bytes
  p.c_vec_ok = ((reinterpret_cast<uintptr_t>(a.C) & 15u) == 0 && (a.ldc % VEC) == 0 &&
                (a.batch <= 1 || (a.stride_c % VEC) == 0)) ? 1 : 0;
  p.c_tma = (p.c_vec_ok && a.splits <= 1 && a.c_tma &&
             bn >= (sizeof(T) == 4 ? 32 : 64)) ? 1 : 0;
  p.pair = hgemm_use_pair(bn, a.M, p.splits, a.pair) ? a.pair : 0;
  p.dp_units = a.dp_units;
  p.tail_splits = a.tail_splits;
  p.tail_k_slice = a.tail_k_slice;
  p.tail_ws = a.tail_ws;
  p.tail_cnt = a.tail_cnt;
  p.batch = a.batch > 1 ? a.batch : 1;
  p.stride_c = p.batch > 1 ? a.stride_c : 0;
  p.za_mask = (p.batch > 1 && a.stride_a != 0) ? -1 : 0;
  p.ep = a.ep;
  // Short-K tiles are epilogue-bound: both shares of epilogue warps drain them
  // (measured: 4096 x 4096 x 128 fp16 23.2 -> 19-21 us); long-K tiles keep one
  // share, which leaves the main loop's warps more issue slots (4096^3 and
  // 8192^3 were 2 % slower with two).
  {
    const int steps = (p.k_slice + kblk<T>() - 1) / kblk<T>();
    p.epi_halves = (EPI_HALVES > 1 && steps <= 8) ? EPI_HALVES : 1;
  }
  p.zb_mask = (p.batch > 1 && a.stride_b != 0) ? -1 : 0;
  if (p.tail_splits > 0 && (p.splits != 1 || !p.tail_ws || !p.tail_cnt)) return cudaErrorInvalidValue;
  if (p.batch > 1 && (p.splits != 1 || p.tail_splits > 0)) return cudaErrorInvalidValue;
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
