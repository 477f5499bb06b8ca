// Host-side declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gb300 {

// One fp32 GEMM launch over a K range per grid z-slice.
// Fused epilogue of a GEMM: C = act(alpha * AB + beta * C + bias[j]).
// bias: N elements of the output type (device), or null; act: 0 none, 1 relu,
// 2 gelu.
struct Epilogue {
  const void* bias = nullptr;
  int act = 0;
};

struct SgemmArgs {
  int transA, transB;
  int M, N, K;
  const float* A;
  int64_t lda;
  const float* B;
  int64_t ldb;
  float* C;
  int64_t ldc;
  float alpha, beta;
  // split-K: slice z covers k in [z*k_slice, min(K, (z+1)*k_slice)); when
  // splits > 1 the kernel writes raw sums to partial[z][M][N] instead of C.
  int splits;
  int k_slice;
  float* partial;
  // strided batch (batch > 1, at most 65535, no split): matrix y of the batch
  // is A + y*stride_a, B + y*stride_b, C + y*stride_c (elements)
  int batch = 1;
  int64_t stride_a = 0, stride_b = 0, stride_c = 0;
  // persistent stream-K launch (sk_blocks > 0, no split, no batch, at least
  // sk_blocks tiles; not the narrow tile): sk_blocks blocks, partial tiles in
  // sk_ws (sk_blocks * 2 * bm * bn floats of the tile's shape), arrival
  // counters in sk_cnt (one per tile, zero at launch)
  int sk_blocks = 0;
  float* sk_ws = nullptr;
  unsigned int* sk_cnt = nullptr;
  // block tile (SG_TILE_*): the general 128 x 128 tile, the narrow one for
  // N <= SGN_BN, the big 128 x 256 or the half 128 x 64
  int tile = 0;
  // operands k-major (A [K,M], B [K,N]) with 16-byte aligned rows, one GEMM,
  // no split: stage them with the warp-specialised TMA kernel (ws = 1)
  int ws = 0;
  int fault_injection = 0;  // test hook of that kernel (see sgemm_ffma.cuh)
  Epilogue ep;  // fused bias / activation (not with splits > 1: the reduction applies it)
};

// Schedule of one tcgen05 GEMM launch (hgemm_plan): a persistent grid of
// `workers` blocks, or block pairs with pair == 2, over `tiles` output tiles
// of `steps` K steps each.  Tiles [0, dp_tiles) are whole units handed out
// round-robin; the K steps of the others are shared out in sk_workers equal
// contiguous ranges (stream-K), a tile shared by several ranges being summed
// from fp32 partials by its last contributor.
struct HPlan {
  int bn = 0;                 // tile width
  int pair = 0;               // 0 single blocks, 2 two-SM pairs
  int workers = 0;            // blocks (or pairs) in the grid
  int tiles = 0, steps = 0;   // work tiles (batch included), K steps per tile
  int dp_tiles = 0;           // whole tiles
  int sk_workers = 0;         // ranges of the shared steps (0: no sharing)
  int64_t sk_steps = 0;       // (tiles - dp_tiles) * steps
  int sk_publish = 0;         // 1: every contributor publishes; a reduction kernel finishes
  int epi_halves = 1;         // epilogue warps per accumulator quarter
  size_t ws_bytes = 0;        // fp32 partial slots: sk_workers x 2 x (pair ? 2 : 1) x 128 x bn
  size_t cnt_bytes = 0;       // arrival counters, zero before the launch
};

// One tcgen05 GEMM launch (fp16, bf16, or fp32 on TF32 MMAs).
struct HgemmArgs {
  int transA, transB;
  int M, N, K;
  const void* A;  // 16-byte aligned base, row pitch a multiple of 16 bytes
  int64_t lda;
  const void* B;
  int64_t ldb;
  void* C;
  int64_t ldc;
  float alpha, beta;
  int num_sms;
  int bn;               // tile width: 32, 64, 128, 192 or 256
  int c_tma;            // allow TMA stores (and, beta != 0, TMA loads) of C when C is aligned
  int fault_injection;  // test hook: 1 = producer skips its first stage
  int dtype = 1;        // 1 fp16, 2 bf16, 3 fp32 on TF32 MMAs (gemm_dtype_t)
  // 3xTF32 (fp32 operands only): A and B are two planes each, hi and lo, a
  // plane pitch stride_a / stride_b apart; every K step is run three times:
  // hi(A) hi(B), hi(A) lo(B), lo(A) hi(B)
  int split3 = 0;
  // strided batch (batch > 1): element pitches between consecutive matrices;
  // 16-bit TMA needs them (and ld) multiples of 8
  int batch = 1;
  int64_t stride_a = 0, stride_b = 0, stride_c = 0;
  HPlan plan;                      // from hgemm_plan
  float* sk_ws = nullptr;          // plan.ws_bytes of scratch when plan.sk_workers > 0
  unsigned int* sk_cnt = nullptr;  // plan.cnt_bytes, zeroed before the launch
  Epilogue ep;  // fused bias / activation
};

struct LaunchCtx {
  cudaStream_t stream;
  unsigned int* status;  // device status word
  uint64_t timeout_ns;
  int launches;          // incremented per kernel launched
  int grid = 0;          // blocks of the last main GEMM kernel launched
};

// Launchers (return cudaSuccess or the launch error).
// Programmatic dependent launch of the library's kernels (env GEMM_GB300_PDL=0
// turns it off).
int pdl_enabled();

cudaError_t launch_sgemm(const SgemmArgs& a, LaunchCtx& ctx);
cudaError_t launch_sgemm_narrow(const SgemmArgs& a, LaunchCtx& ctx);  // SG_TILE_NARROW
cudaError_t launch_sgemm_big(const SgemmArgs& a, LaunchCtx& ctx);     // SG_TILE_BIG
cudaError_t launch_sgemm_half(const SgemmArgs& a, LaunchCtx& ctx);    // SG_TILE_HALF
cudaError_t launch_hgemm(const HgemmArgs& a, LaunchCtx& ctx);
cudaError_t launch_hgemm_bf16(const HgemmArgs& a, LaunchCtx& ctx);
// fp32 operands and output on kind::tf32 MMAs (HgemmArgs.dtype 3; K-major A and B)
cudaError_t launch_hgemm_tf32(const HgemmArgs& a, LaunchCtx& ctx);
// C[M,N] = alpha * sum_z P[z] + beta * C; dtype 0 = fp32 C, 1 = fp16 C, 2 = bf16 C.
cudaError_t launch_splitk_reduce(int dtype, int M, int N, int splits, const float* P, void* C,
                                 int64_t ldc, float alpha, float beta, LaunchCtx& ctx,
                                 Epilogue ep = Epilogue());
// C = act(beta * C + bias) (K == 0); beta == 0 reads no C.
cudaError_t launch_scale(int dtype, int M, int N, void* C, int64_t ldc, float beta,
                         LaunchCtx& ctx, Epilogue ep = Epilogue());
// 3xTF32 operand split: hi = the TF32 part of each fp32 value (low 13
// fraction bits cleared), lo = x - hi (exact), into two planes of row pitch
// ld_dst (a multiple of 4, 16-byte aligned).  transpose == false: planes
// [rows][cols] from src [rows][cols], padding columns zeroed; true: planes
// [cols][rows] from src [rows][cols], padding not written.
cudaError_t launch_split_tf32(bool transpose, int rows, int cols, const float* src,
                              int64_t ld_src, float* hi, float* lo, int64_t ld_dst,
                              LaunchCtx& ctx);
// dst[c][r] = src[r][c] (fp32 rows x cols).
cudaError_t launch_transpose_f32(int rows, int cols, const float* src, int64_t ld_src,
                                 float* dst, int64_t ld_dst, LaunchCtx& ctx);
// dst[r][c] = src[r][c] for c < cols, 0 for cols <= c < ld_dst, into a dst
// with 16-byte aligned rows (base 16-byte aligned, ld_dst a multiple of 4
// elements for repack_32 or 8 for repack_16; else cudaErrorInvalidValue).
// 32-bit or 16-bit elements (fp16 or bf16: +0 is the zero bit pattern in both).
cudaError_t launch_repack_32(int rows, int cols, const void* src, int64_t ld_src, void* dst,
                             int64_t ld_dst, LaunchCtx& ctx);
cudaError_t launch_repack_16(int rows, int cols, const void* src, int64_t ld_src, void* dst,
                             int64_t ld_dst, LaunchCtx& ctx);
// dst[r][c] = src[r][c] for c < cols, any alignment on either side (element
// size 2 or 4 bytes): the way back from an aligned scratch copy of C.
cudaError_t launch_copy_rows(int esize, int rows, int cols, const void* src, int64_t ld_src,
                             void* dst, int64_t ld_dst, LaunchCtx& ctx);

// Tile sizes the dispatcher needs.
// fp32 block tile: (64 * SG_WARPS_M) x SG_BN, K step SG_BK, SG_BLOCKS_PER_SM
// resident blocks per SM (compile-time knobs; the defaults measured fastest)
#ifndef GB300_SG_WARPS_M
#define GB300_SG_WARPS_M 2
#endif
constexpr int SG_WARPS_M = GB300_SG_WARPS_M;
#ifndef GB300_SG_BK
#define GB300_SG_BK 64
#endif
#ifndef GB300_SG_BN
#define GB300_SG_BN 128
#endif
#ifndef GB300_SG_MIN_BLOCKS
#define GB300_SG_MIN_BLOCKS 1
#endif
constexpr int SG_BM = 64 * SG_WARPS_M, SG_BN = GB300_SG_BN, SG_BK = GB300_SG_BK;
constexpr int SG_BLOCKS_PER_SM = GB300_SG_MIN_BLOCKS;
// fp32 narrow tile for N <= 32: a 128 x 128 tile would leave 3/4 of its
// columns idle (the rank-32 output of a LoRA projection, M=8192 N=32 K=8192)
#ifndef GB300_SGN_WARPS_M
#define GB300_SGN_WARPS_M 4
#endif
#ifndef GB300_SGN_BK
#define GB300_SGN_BK 32
#endif
#ifndef GB300_SGN_MIN_BLOCKS
#define GB300_SGN_MIN_BLOCKS 2
#endif
// (stages of its ring: three at two blocks per SM; two stages at three
// blocks per SM measured level or slower: 512 x 32 x 5632 nn kernel 23.2 ->
// 25.2 us, 8192 x 32 x 8192 88.7 us either way)
#ifndef GB300_SGN_STAGES
#define GB300_SGN_STAGES 3
#endif
constexpr int SGN_BM = 64 * GB300_SGN_WARPS_M, SGN_BN = 32, SGN_BK = GB300_SGN_BK;
constexpr int SGN_BLOCKS_PER_SM = GB300_SGN_MIN_BLOCKS;
constexpr int SGN_STAGES = GB300_SGN_STAGES;
// fp32 big tile: 128 x 256 at K step 32 in a 4-stage ring, one block of 8
// warps per SM, each lane 8 rows x 16 columns -- per K a lane builds its 8
// splatted A pairs once for 64 paired FMAs (32 with 8 x 8), and the block
// reads 3/8 rather than 1/2 a float from shared memory per FMA pair
constexpr int SGB_BM = 128, SGB_BN = 256, SGB_BK = 32, SGB_STAGES = 4;
// fp32 half tile: 128 x 64 at K step 32 in a 4-stage ring, 4 warps, two
// blocks per SM: twice the tiles of 128 x 128 for grids that leave SMs idle
constexpr int SGH_BM = 128, SGH_BN = 64, SGH_BK = 32, SGH_STAGES = 4, SGH_BLOCKS_PER_SM = 2;
// fp32 tile ids (SgemmArgs::tile) and their shapes
enum { SG_TILE_WIDE = 0, SG_TILE_NARROW = 1, SG_TILE_BIG = 2, SG_TILE_HALF = 3 };
struct SgTileShape {
  int bm, bn, bk, blocks_per_sm;
};
inline SgTileShape sg_tile_shape(int tile) {
  switch (tile) {
    case SG_TILE_NARROW: return {SGN_BM, SGN_BN, SGN_BK, SGN_BLOCKS_PER_SM};
    case SG_TILE_BIG: return {SGB_BM, SGB_BN, SGB_BK, 1};
    case SG_TILE_HALF: return {SGH_BM, SGH_BN, SGH_BK, SGH_BLOCKS_PER_SM};
    default: return {SG_BM, SG_BN, SG_BK, SG_BLOCKS_PER_SM};
  }
}
constexpr int HG_BM = 128, HG_BK = 64;
// Tile width of the tcgen05 kernel (32 to 256 columns) for this problem and
// schedule (arguments as hgemm_plan).
int hgemm_pick_bn(int M, int N, int K, int transA, int transB, int kstep, int batch,
                  int pair_allowed, int num_sms, int sk_mode);
bool hgemm_use_pair(int bn, int M, int allowed);
int hgemm_pair_slots(int bn, int transA, int transB, int num_sms);
// Schedule of a tcgen05 launch.  kstep: K elements per step (64 for 16-bit
// operands, 32 for TF32); pair_allowed: 0 or 2; sk_mode: 0 whole tiles only,
// 1 share K steps when that pays (the last one or two rounds of tiles,
// finished inside the kernel; or, with fewer tiles than workers, every tile,
// finished by a reduction kernel), 2 share every tile and finish inside the
// kernel, 3 share every tile and finish with the reduction kernel (2 and 3
// are test settings).
HPlan hgemm_plan(int M, int N, int K, int bn, int transA, int transB, int kstep, int batch,
                 int pair_allowed, int num_sms, int sk_mode);

}  // namespace gb300
