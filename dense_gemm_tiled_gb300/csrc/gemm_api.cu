// The C ABI (include/gemm.h): argument checks, variant canonicalisation,
// kernel-path choice, scratch management, launch, device status.
//
// Path choice:
//   dtype fp32 -> CUDA-core FFMA kernel (sgemm_ffma.cu); split-K when the
//                 output has too few tiles to fill the GPU.
//   dtype fp16 / bf16 -> tcgen05 kernel (hgemm_tcgen05.cuh); split-K likewise.
// The split-K rule follows "Metal GEMM Kernels for LoRA Training", section 5
// (route by output-tile count; fp32 partials in device memory, then a
// reduction), with the threshold set by this GPU's SM count instead of the
// page's fixed 32 tiles, and with K slices that need not divide K evenly.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <memory>
#include <mutex>

#include "../../include/gemm.h"
#include "internal.h"

using namespace gb300;

namespace gb300 {
// Programmatic dependent launch switch (declared in internal.h).
int pdl_enabled() {
  static const int v = [] {
    const char* e = getenv("GEMM_GB300_PDL");
    return e ? atoi(e) : 1;
  }();
  return v;
}
}  // namespace gb300

namespace {

__device__ unsigned int g_status_word;  // per device: bits of STATUS_*

constexpr int MAX_DEVICES = 64;
std::mutex g_mu;
unsigned int* g_status_ptr[MAX_DEVICES];
int g_num_sms[MAX_DEVICES];
std::atomic<int64_t> g_total_launches{0};
std::atomic<int64_t> g_timeout_ns{2000000000LL};
std::atomic<int> g_fault_injection{0};
thread_local int tl_last_path = GEMM_PATH_NONE;
thread_local int tl_last_launches = 0;
thread_local int tl_last_grid = 0;
// gemm_set_kernel_events: recorded around the main GEMM kernel of each call
thread_local cudaEvent_t tl_ev_start = nullptr, tl_ev_end = nullptr;

// The main GEMM kernel launch, bracketed by the caller's timing events when
// set.
cudaError_t timed_sgemm(const SgemmArgs& a, LaunchCtx& ctx) {
  if (tl_ev_start && tl_ev_end) {
    cudaError_t e = cudaEventRecord(tl_ev_start, ctx.stream);
    if (e != cudaSuccess) return e;
    e = launch_sgemm(a, ctx);
    if (e != cudaSuccess) return e;
    return cudaEventRecord(tl_ev_end, ctx.stream);
  }
  return launch_sgemm(a, ctx);
}
cudaError_t timed_hgemm(const HgemmArgs& a, LaunchCtx& ctx) {
  if (tl_ev_start && tl_ev_end) {
    cudaError_t e = cudaEventRecord(tl_ev_start, ctx.stream);
    if (e != cudaSuccess) return e;
    e = launch_hgemm(a, ctx);
    if (e != cudaSuccess) return e;
    return cudaEventRecord(tl_ev_end, ctx.stream);
  }
  return launch_hgemm(a, ctx);
}

// Per-device set-up, done once with that device current: the status word's
// device address and the SM count.
int device_state(int* dev_out, unsigned int** status, int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_CUDA;
  if (dev < 0 || dev >= MAX_DEVICES) return GEMM_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return GEMM_ERR_CUDA;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return GEMM_ERR_CUDA;
    g_num_sms[dev] = n > 0 ? n : 1;
    g_status_ptr[dev] = static_cast<unsigned int*>(p);
  }
  *dev_out = dev;
  *status = g_status_ptr[dev];
  *sms = g_num_sms[dev];
  return GEMM_OK;
}

// Bytes per element of a gemm_dtype_t, and the output kind the auxiliary
// kernels take (0 fp32, 1 fp16, 2 bf16).
inline bool is_f32(int dtype) {
  return dtype == GEMM_F32 || dtype == GEMM_F32_TF32 || dtype == GEMM_F32_3XTF32;
}
inline int64_t esize(int dtype) { return is_f32(dtype) ? 4 : 2; }
inline int out_kind(int dtype) { return is_f32(dtype) ? 0 : dtype; }

inline int64_t footprint_bytes(int64_t rows, int64_t cols, int64_t ld, int64_t e) {
  if (rows <= 0 || cols <= 0) return 0;
  return ((rows - 1) * ld + cols) * e;
}

inline bool overlaps(const void* a, int64_t na, const void* b, int64_t nb) {
  if (na <= 0 || nb <= 0) return false;
  const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
  return a0 < b0 + (uintptr_t)nb && b0 < a0 + (uintptr_t)na;
}

// Checks shared by gemm() and gemm_host().  Sets the stored shapes of A and B.
int check_args(int transA, int transB, int64_t M, int64_t N, int64_t K, int dtype,
               const void* A, int64_t lda, const void* B, int64_t ldb, const void* C,
               int64_t ldc, int64_t* a_rows, int64_t* a_cols, int64_t* b_rows,
               int64_t* b_cols) {
  if ((transA != 0 && transA != 1) || (transB != 0 && transB != 1)) return GEMM_ERR_INVALID_ARG;
  if (dtype != GEMM_F32 && dtype != GEMM_F16_F32ACC && dtype != GEMM_BF16_F32ACC &&
      dtype != GEMM_F32_TF32 && dtype != GEMM_F32_3XTF32)
    return GEMM_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
  const int64_t lim = (int64_t)1 << 31;
  if (M >= lim || N >= lim || K >= lim) return GEMM_ERR_UNSUPPORTED;
  *a_rows = transA ? K : M;
  *a_cols = transA ? M : K;
  *b_rows = transB ? N : K;
  *b_cols = transB ? K : N;
  if (ldc < (N > 1 ? N : 1)) return GEMM_ERR_INVALID_ARG;
  if (lda < (*a_cols > 1 ? *a_cols : 1)) return GEMM_ERR_INVALID_ARG;
  if (ldb < (*b_cols > 1 ? *b_cols : 1)) return GEMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return GEMM_OK;
  const int64_t e = esize(dtype);
  if (!C || ((uintptr_t)C % (uintptr_t)e) != 0) return GEMM_ERR_INVALID_ARG;
  if (K > 0) {
    if (!A || !B) return GEMM_ERR_INVALID_ARG;
    if (((uintptr_t)A % (uintptr_t)e) != 0 || ((uintptr_t)B % (uintptr_t)e) != 0)
      return GEMM_ERR_INVALID_ARG;
    const int64_t nc = footprint_bytes(M, N, ldc, e);
    if (overlaps(C, nc, A, footprint_bytes(*a_rows, *a_cols, lda, e)) ||
        overlaps(C, nc, B, footprint_bytes(*b_rows, *b_cols, ldb, e)))
      return GEMM_ERR_ALIAS;
  }
  return GEMM_OK;
}

// gemm_host's copy/compute overlap (env GEMM_GB300_HOST_PIPELINE=0 turns it
// off).
int host_pipeline_enabled() {
  static const int v = [] {
    const char* s = getenv("GEMM_GB300_HOST_PIPELINE");
    return (s && s[0] == '0') ? 0 : 1;
  }();
  return v;
}

// gemm_host's schedule on large problems (env GEMM_GB300_HOST_SCHED="P,S,T"):
// P row panels, the first run as S products over K slices (fp32 C), the last
// cut into T pieces so that the final read-back is short.  Zero fields take
// the defaults.
struct HostSched {
  int panels, kslices, tail;
};
HostSched host_sched_env() {
  static const HostSched v = [] {
    HostSched h{0, 0, 0};
    const char* s = getenv("GEMM_GB300_HOST_SCHED");
    if (s) sscanf(s, "%d,%d,%d", &h.panels, &h.kslices, &h.tail);
    return h;
  }();
  return v;
}

// fp32 stream-K persistent launch (env GEMM_GB300_SG_SK=0 turns it off).
int sg_sk_enabled() {
  static const int v = [] {
    const char* s = getenv("GEMM_GB300_SG_SK");
    return (s && s[0] == '0') ? 0 : 1;
  }();
  return v;
}

// fp32 packing pre-pass (env GEMM_GB300_SG_PACK=0 turns it off).
int sg_pack_enabled() {
  static const int v = [] {
    const char* e = getenv("GEMM_GB300_SG_PACK");
    return e ? atoi(e) : 1;
  }();
  return v;
}

// fp32 narrow tile for N <= 32 (env GEMM_GB300_SG_NARROW=0 turns it off).
int sg_narrow_enabled() {
  static const int v = [] {
    const char* e = getenv("GEMM_GB300_SG_NARROW");
    return e ? atoi(e) : 1;
  }();
  return v;
}

// fp32 tile for N > 32 (env GEMM_GB300_SG_TILE): 0 the 128 x 128 tile, 2 the
// 128 x 256 one, 3 the 128 x 64 one; unset or any other value: the
// dispatcher's choice.
int sg_tile_forced() {
  static const int v = [] {
    const char* e = getenv("GEMM_GB300_SG_TILE");
    const int t = e ? atoi(e) : -1;
    return (t == SG_TILE_WIDE || t == SG_TILE_BIG || t == SG_TILE_HALF) ? t : -1;
  }();
  return v;
}

// fp32 warp-specialised TMA staging for k-major aligned operands (env
// GEMM_GB300_SG_WS=0 turns it off).
int sg_ws_enabled() {
  static const int v = [] {
    const char* e = getenv("GEMM_GB300_SG_WS");
    return (e && e[0] == '0') ? 0 : 1;
  }();
  return v;
}

// fp16 block pairs (env GEMM_GB300_HG_PAIR): 0 single blocks, 2 (default)
// pairs running 2-SM (cta_group::2) MMAs; any other value means 2.
int pair_enabled() {
  static const int v = [] {
    const char* e = getenv("GEMM_GB300_HG_PAIR");
    return (e && atoi(e) == 0) ? 0 : 2;
  }();
  return v;
}

// Debug/bench switch for the fp16 TMA-store epilogue (env GEMM_GB300_HG_CTMA=0
// turns it off).
int c_tma_enabled() {
  static const int v = [] {
    const char* e = getenv("GEMM_GB300_HG_CTMA");
    return e ? atoi(e) : 1;
  }();
  return v;
}

// A C whose rows are not 16-byte aligned cannot go through the tensor-memory-
// access unit; the tensor-core kernel then stores it row by row through its
// staging buffers, which on large problems costs more than computing into an
// aligned scratch copy (TMA stores, and TMA loads when beta != 0) and moving
// that into place with a copy kernel (measured 4095^3 fp16, whole call:
// 170 us row by row against 155 us through the copy with beta = 0, 335 us
// against 177 us with beta = 1).
bool c_scratch_wanted(const void* C, int64_t ldc, int64_t es, int M, int N) {
  const bool aligned = ((uintptr_t)C % 16) == 0 && (ldc * es) % 16 == 0;
  return !aligned && c_tma_enabled() && (int64_t)M * N >= (1ll << 21);
}

// Stream-K schedule of the tensor-core kernel (env GEMM_GB300_HG_SK): 1
// (default) shares out K steps when that pays; 0 whole tiles only; 2 and 3
// share every tile, finished inside the kernel (2) or by the reduction kernel
// (3) -- test settings that force those paths.
int sk_mode() {
  static const int v = [] {
    const char* e = getenv("GEMM_GB300_HG_SK");
    const int m = e ? atoi(e) : 1;
    return (m >= 0 && m <= 3) ? m : 1;
  }();
  return v;
}

// Debug/bench override of the fp16 tile width (env GEMM_GB300_HG_BN); 0 = the
// dispatcher's own choice.
int forced_bn() {
  static const int v = [] {
    const char* e = getenv("GEMM_GB300_HG_BN");
    return e ? atoi(e) : 0;
  }();
  return v;
}

// Tile width of the tensor-core kernel for 16-bit operands: the dispatcher's
// model, unless GEMM_GB300_HG_BN forces one (32 only for a K-major B with
// N <= 32).
int pick_bn16(int M, int N, int K, int transA, int transB, int sms, int batch, int skm) {
  int bn = hgemm_pick_bn(M, N, K, transA, transB, HG_BK, batch, pair_enabled(), sms, skm);
  const int forced = forced_bn();
  if (forced == 32 ? (N <= 32 && transB)
                   : (forced == 64 || forced == 128 || forced == 192 || forced == 256))
    bn = forced;
  return bn;
}

int cuda_fail(cudaError_t e) { return e == cudaErrorMemoryAllocation ? GEMM_ERR_NO_MEMORY : GEMM_ERR_CUDA; }

// fp32 problem size (M*N*K, as a power of two) from which operands are packed
// into the layout the kernels read fastest, and the most contributors a tile
// gets when every tile's K steps are shared (resident blocks / tiles), as
// compile-time knobs.  Measured on GB300 (whole calls, L2 flushed): packing
// from 2^27 lost where it changed the path (1024 x 1024 x 512 38.6 -> 41.7 us,
// 768 x 1024 x 768 nt 41.7 -> 46.1 us); up to 8 contributors against 4 gained
// on 30 to 37 tiles (640 x 640 x 16384 265 -> 226 us, 768 x 768 x 8192 196 ->
// 169 us, 640 x 768 x 4096 95 -> 85 us).
#ifndef GB300_SG_PACK_MIN_LOG2
#define GB300_SG_PACK_MIN_LOG2 30
#endif
#ifndef GB300_SG_SKALL_MAX_SHARE
#define GB300_SG_SKALL_MAX_SHARE 8
#endif
constexpr double SG_PACK_MIN = (double)(1ll << GB300_SG_PACK_MIN_LOG2);

// Split-K plan of the fp32 kernel: how many K slices, each a multiple of
// `kstep` long.  Fewest K steps a slice gets (compile-time knob): one (a
// 64-deep step of a 128 x 128 tile is ~1M FMAs), measured on small squares
// against 2 and 4: 256^3 16 / 21 / 31 us, 512^3 18 / 23 / 33 us.
#ifndef GB300_SG_SLICE_STEPS
#define GB300_SG_SLICE_STEPS 1
#endif

void plan_splits(int64_t tiles, int64_t K, int kstep, int capacity, int min_steps_per_slice,
                 int max_splits, int* splits, int* k_slice) {
  const int64_t steps = (K + kstep - 1) / kstep;
  int s = 1;
  if (tiles * 2 <= capacity && steps >= 2 * min_steps_per_slice) {
    int64_t want = capacity / (tiles > 0 ? tiles : 1);
    int64_t cap_k = steps / min_steps_per_slice;
    int64_t ss = want < cap_k ? want : cap_k;
    if (ss > max_splits) ss = max_splits;
    s = ss > 1 ? (int)ss : 1;
  }
  if (s <= 1) {
    *splits = 1;
    *k_slice = (int)(steps * kstep);
    return;
  }
  const int64_t per = (steps + s - 1) / s;  // steps per slice
  *k_slice = (int)(per * kstep);
  *splits = (int)((steps + per - 1) / per);  // every slice non-empty
}

// fp32 tile and K split: N <= 32 takes the narrow tile (256 x 32, two blocks
// per SM), split over K until one round of resident blocks is full; other
// shapes the 128 x 128 tile, split when the tiles fill under half of two
// rounds of the SMs.
void plan_f32(int M, int N, int K, int sms, int* tile, int64_t* tiles, int* splits,
              int* k_slice) {
  if (N <= SGN_BN && sg_narrow_enabled()) *tile = SG_TILE_NARROW;
  else if (sg_tile_forced() >= 0) *tile = sg_tile_forced();
  else *tile = SG_TILE_WIDE;
  const SgTileShape ts = sg_tile_shape(*tile);
  *tiles = (int64_t)((M + ts.bm - 1) / ts.bm) * ((N + ts.bn - 1) / ts.bn);
  if (*tile == SG_TILE_NARROW)
    plan_splits(*tiles, K, SGN_BK, sms * SGN_BLOCKS_PER_SM, 8, 16, splits, k_slice);
  else
    plan_splits(*tiles, K, ts.bk, 2 * sms * ts.blocks_per_sm, GB300_SG_SLICE_STEPS, 16, splits,
                k_slice);
}

// Scratch comes from a stream-ordered memory pool owned by the library, one
// per device, that keeps freed memory for reuse (release threshold: never).
// The device's default pool would hand its memory back at every
// synchronisation, and re-mapping a few MB costs ~0.1 ms per call.
cudaMemPool_t g_pool[MAX_DEVICES];

cudaError_t scratch_pool(cudaMemPool_t* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_pool[dev]) {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool;
    e = cudaMemPoolCreate(&pool, &props);
    if (e != cudaSuccess) return e;
    uint64_t keep = UINT64_MAX;
    e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
    if (e != cudaSuccess) return e;
    g_pool[dev] = pool;
  }
  *out = g_pool[dev];
  return cudaSuccess;
}

inline size_t pad256(size_t n) { return (n + 255) / 256 * 256; }

struct Scratch {
  void* ptr = nullptr;
  cudaStream_t stream = nullptr;
  ~Scratch() {
    if (ptr) cudaFreeAsync(ptr, stream);
  }
  cudaError_t get(size_t bytes, cudaStream_t s) {
    stream = s;
    cudaMemPool_t pool;
    cudaError_t e = scratch_pool(&pool);
    if (e != cudaSuccess) return e;
    return cudaMallocFromPoolAsync(&ptr, bytes, pool, s);
  }
};

int run_gemm(int transA, int transB, int64_t M64, int64_t N64, int64_t K64, int dtype,
             float alpha, float beta, const void* A, int64_t lda, const void* B, int64_t ldb,
             void* C, int64_t ldc, cudaStream_t stream, int64_t a_rows, int64_t a_cols,
             int64_t b_rows, int64_t b_cols, Epilogue ep = Epilogue()) {
  int dev, sms;
  unsigned int* status;
  int rc = device_state(&dev, &status, &sms);
  if (rc != GEMM_OK) return rc;
  LaunchCtx ctx{stream, status, (uint64_t)g_timeout_ns.load(), 0};
  const int M = (int)M64, N = (int)N64, K = (int)K64;
  int path = GEMM_PATH_NONE;
  cudaError_t e = cudaSuccess;

  if (K == 0) {
    path = GEMM_PATH_SCALE;
    e = launch_scale(out_kind(dtype), M, N, C, ldc, beta, ctx, ep);
  } else if (dtype == GEMM_F32_TF32 || dtype == GEMM_F32_3XTF32) {
    // Opt-in TF32: the tcgen05 kernel on kind::tf32 reads K-major fp32
    // operands in 16-byte aligned rows, A [M, K] and B [N, K]; others are
    // transposed or re-pitched into scratch first.  3xTF32: every operand is
    // split into TF32 hi and lo planes (K-major, in scratch) and the kernel
    // runs hi*hi + hi*lo + lo*hi over one K loop of three segments.
    const bool x3 = dtype == GEMM_F32_3XTF32;
    const int64_t ldk = (K + 3) / 4 * 4;
    const int steps_k = (K + 31) / 32;
    const int K_eff = x3 ? 3 * steps_k * 32 : K;
    const int bn = hgemm_pick_bn(M, N, K_eff, 0, 1, 32, 1, pair_enabled(), sms, sk_mode());
    const HPlan pl = hgemm_plan(M, N, K_eff, bn, 0, 1, 32, 1, pair_enabled(), sms, sk_mode());
    const bool a_ok = !x3 && !transA && ((uintptr_t)A % 16) == 0 && (lda % 4) == 0;
    const bool b_ok = !x3 && transB && ((uintptr_t)B % 16) == 0 && (ldb % 4) == 0;
    const int planes = x3 ? 2 : 1;
    const size_t bytes_a = a_ok ? 0 : pad256((size_t)planes * M * ldk * 4);
    const size_t bytes_b = b_ok ? 0 : pad256((size_t)planes * N * ldk * 4);
    const size_t bytes_w = pad256(pl.ws_bytes), bytes_n = pad256(pl.cnt_bytes);
    const bool c_scr = c_scratch_wanted(C, ldc, 4, M, N);
    const int64_t ldc_p = (N + 3) / 4 * 4;
    const size_t bytes_c = c_scr ? pad256((size_t)M * ldc_p * 4) : 0;
    Scratch ws;
    const size_t total = bytes_a + bytes_b + bytes_w + bytes_n + bytes_c;
    if (total > 0) {
      e = ws.get(total, stream);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    char* wp = (char*)ws.ptr;
    float* At = (float*)wp;
    float* Bt = (float*)(wp + bytes_a);
    float* sk_ws = (float*)(wp + bytes_a + bytes_b);
    unsigned int* sk_cnt = (unsigned int*)(wp + bytes_a + bytes_b + bytes_w);
    void* Cd = c_scr ? (void*)(wp + bytes_a + bytes_b + bytes_w + bytes_n) : C;
    const int64_t ldcd = c_scr ? ldc_p : ldc;
    if (c_scr && beta != 0.f) e = launch_repack_32(M, N, C, ldc, Cd, ldc_p, ctx);
    if (e == cudaSuccess && pl.cnt_bytes > 0)
      e = cudaMemsetAsync(sk_cnt, 0, pl.cnt_bytes, stream);
    const void* Ad = A;
    const void* Bd = B;
    int64_t ldad = lda, ldbd = ldb;
    if (e == cudaSuccess && x3) {
      // A [M,K] rows, or A [K,M] transposed; B [N,K] rows, or B [K,N] transposed
      e = launch_split_tf32(transA != 0, transA ? K : M, transA ? M : K, (const float*)A, lda, At,
                            At + (int64_t)M * ldk, ldk, ctx);
      if (e == cudaSuccess)
        e = launch_split_tf32(transB == 0, transB ? N : K, transB ? K : N, (const float*)B, ldb,
                              Bt, Bt + (int64_t)N * ldk, ldk, ctx);
      Ad = At; ldad = ldk;
      Bd = Bt; ldbd = ldk;
    } else {
      if (e == cudaSuccess && !a_ok) {
        e = transA ? launch_transpose_f32(K, M, (const float*)A, lda, At, ldk, ctx)
                   : launch_repack_32(M, K, A, lda, At, ldk, ctx);
        Ad = At; ldad = ldk;
      }
      if (e == cudaSuccess && !b_ok) {
        e = !transB ? launch_transpose_f32(K, N, (const float*)B, ldb, Bt, ldk, ctx)
                    : launch_repack_32(N, K, B, ldb, Bt, ldk, ctx);
        Bd = Bt; ldbd = ldk;
      }
    }
    if (e == cudaSuccess) {
      HgemmArgs a{0, 1, M, N, K, Ad, ldad, Bd, ldbd, Cd, ldcd, alpha, beta, sms, bn,
                  c_tma_enabled(), g_fault_injection.load()};
      a.dtype = GEMM_F32_TF32;
      a.plan = pl;
      a.sk_ws = sk_ws;
      a.sk_cnt = sk_cnt;
      a.ep = ep;
      if (x3) {
        a.split3 = 1;
        a.stride_a = (int64_t)M * ldk;  // plane pitches
        a.stride_b = (int64_t)N * ldk;
      }
      path = pl.sk_workers > 0 ? GEMM_PATH_TC_SPLITK : GEMM_PATH_TC;
      e = timed_hgemm(a, ctx);
      if (e == cudaSuccess && c_scr) e = launch_copy_rows(4, M, N, Cd, ldc_p, C, ldc, ctx);
    }
  } else if (dtype == GEMM_F32) {
    int tile, splits, k_slice;
    int64_t tiles;
    plan_f32(M, N, K, sms, &tile, &tiles, &splits, &k_slice);
    const bool narrow = tile == SG_TILE_NARROW;
    const SgTileShape ts = sg_tile_shape(tile);
    const int64_t G = (int64_t)sms * ts.blocks_per_sm;  // resident blocks
    // Fewer tiles than resident blocks on a large problem: rather than K
    // slices and a reduction kernel, the warp-specialised kernel (operands
    // packed k-major) shares every tile's K steps evenly over all blocks in
    // one launch, the last contributor to a tile adding the others' partial
    // sums -- while a tile has at most about GB300_SG_SKALL_MAX_SHARE
    // contributors (its fix-up is one block's reads).  Every block's step
    // range must be non-empty.
    const int64_t kiters = (K + ts.bk - 1) / ts.bk;
    const bool sk_all = splits > 1 && !narrow && sg_ws_enabled() && sg_sk_enabled() &&
                        sg_pack_enabled() && (double)M * N * K >= SG_PACK_MIN &&
                        tiles * GB300_SG_SKALL_MAX_SHARE >= G && tiles * kiters >= G;
    if (sk_all) {
      splits = 1;
      k_slice = K;
    }
    SgemmArgs a{transA, transB, M, N, K, (const float*)A, lda, (const float*)B, ldb, (float*)C,
                ldc, alpha, beta, splits, k_slice, nullptr};
    a.tile = tile;
    a.ws = sg_ws_enabled();
    a.fault_injection = g_fault_injection.load();
    if (splits == 1) a.ep = ep;  // split-K: the reduction applies it
    // Packing: the kernel reads A stored [K,M] and B stored [K,N] fastest
    // (measured at 4096^3: tn 56.4 TF/s, nn 53.7, nt 46.9), so on large
    // problems an operand stored with k contiguous is first transposed into
    // that layout (HBM-bound, ~1 % of the GEMM's time at 4096^3).
    // An operand whose rows are not 16-byte aligned is read with 4-byte
    // copies (measured 4095^3: 42 TF/s); on large problems it is copied into
    // a padded row pitch first, so the kernel takes 16-byte copies throughout.
    // (The narrow tile streams A once with no reuse across tile columns, so
    // transposing A would double its traffic: only a misaligned operand is
    // copied there, and it splits over K, so the test is on the problem size.)
    const bool big = (splits == 1 || narrow) && sg_pack_enabled() &&
                     (double)M * N * K >= SG_PACK_MIN;
    auto misaligned = [](const void* p, int64_t ld) { return ((uintptr_t)p % 16) != 0 || ld % 4 != 0; };
    const bool packA = big && ((!transA && !narrow) || misaligned(A, lda));
    const bool packB = big && (transB || misaligned(B, ldb));
    const int64_t ldA_p = (M + 3) / 4 * 4, ldB_p = (N + 3) / 4 * 4, ldK_p = (K + 3) / 4 * 4;
    const bool a_rows = narrow && !transA;  // A copied as [M,K] rows, not transposed
    const size_t bytes_A =
        packA ? ((size_t)(a_rows ? M * ldK_p : K * ldA_p) * 4 + 255) / 256 * 256 : 0;
    const size_t bytes_B = packB ? ((size_t)K * ldB_p * 4 + 255) / 256 * 256 : 0;
    const size_t bytes_P = splits > 1 ? (size_t)splits * M * N * sizeof(float) : 0;
    // Stream-K: without a split, a tile count that is not a whole number of
    // rounds of the SMs leaves the last round part-empty (4096^3: 1024 tiles,
    // 6.7 rounds of 152).  The persistent launch gives whole tiles to all but
    // the last one to two rounds and shares those rounds' K steps evenly.
    const bool sk = splits == 1 && !narrow && sg_sk_enabled() && tiles % G != 0 &&
                    (tiles >= G || sk_all);
    const int64_t sk_tiles = sk ? (tiles >= 2 * G ? tiles % G + G : tiles) : 0;
    const size_t bytes_S = sk ? (size_t)G * 2 * ts.bm * ts.bn * sizeof(float) : 0;
    const size_t bytes_N = sk ? ((size_t)sk_tiles * sizeof(unsigned int) + 255) / 256 * 256 : 0;
    Scratch ws;
    if (bytes_A + bytes_B + bytes_P + bytes_S + bytes_N > 0) {
      e = ws.get(bytes_A + bytes_B + bytes_P + bytes_S + bytes_N, stream);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    if (splits > 1) a.partial = (float*)((char*)ws.ptr + bytes_A + bytes_B);
    if (sk) {
      a.sk_blocks = (int)G;
      a.sk_ws = (float*)((char*)ws.ptr + bytes_A + bytes_B + bytes_P);
      a.sk_cnt = (unsigned int*)((char*)a.sk_ws + bytes_S);
      e = cudaMemsetAsync(a.sk_cnt, 0, (size_t)sk_tiles * sizeof(unsigned int), stream);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    if (packA && a_rows) {  // A [M,K] into an aligned pitch
      float* At = (float*)ws.ptr;
      e = launch_repack_32(M, K, A, lda, At, ldK_p, ctx);
      a.A = At; a.lda = ldK_p;
    } else if (packA) {  // A [M,K] -> [K,M], or A [K,M] into an aligned pitch
      float* At = (float*)ws.ptr;
      e = transA ? launch_repack_32(K, M, A, lda, At, ldA_p, ctx)
                 : launch_transpose_f32(M, K, (const float*)A, lda, At, ldA_p, ctx);
      a.A = At; a.lda = ldA_p; a.transA = 1;
    }
    if (e == cudaSuccess && packB) {  // B [N,K] -> [K,N], or B [K,N] into an aligned pitch
      float* Bt = (float*)((char*)ws.ptr + bytes_A);
      e = transB ? launch_transpose_f32(N, K, (const float*)B, ldb, Bt, ldB_p, ctx)
                 : launch_repack_32(K, N, B, ldb, Bt, ldB_p, ctx);
      a.B = Bt; a.ldb = ldB_p; a.transB = 0;
    }
    path = splits > 1 ? GEMM_PATH_FFMA_SPLITK : GEMM_PATH_FFMA;
    if (e == cudaSuccess) e = timed_sgemm(a, ctx);
    if (e == cudaSuccess && splits > 1)
      e = launch_splitk_reduce(0, M, N, splits, a.partial, C, ldc, alpha, beta, ctx, ep);
  } else {
    const int bn = pick_bn16(M, N, K, transA, transB, sms, 1, sk_mode());
    const HPlan pl = hgemm_plan(M, N, K, bn, transA, transB, HG_BK, 1, pair_enabled(), sms,
                                sk_mode());
    // The tensor-memory-access unit needs 16-byte aligned bases and row
    // pitches; an operand that has neither is copied into padded scratch.
    const bool a_ok = ((uintptr_t)A % 16) == 0 && (lda % 8) == 0;
    const bool b_ok = ((uintptr_t)B % 16) == 0 && (ldb % 8) == 0;
    const int64_t lda_p = (a_cols + 7) / 8 * 8, ldb_p = (b_cols + 7) / 8 * 8;
    const size_t bytes_a = a_ok ? 0 : pad256((size_t)(a_rows * lda_p * 2));
    const size_t bytes_b = b_ok ? 0 : pad256((size_t)(b_rows * ldb_p * 2));
    const size_t bytes_w = pad256(pl.ws_bytes), bytes_n = pad256(pl.cnt_bytes);
    // C rows not 16-byte aligned: see c_scratch_wanted
    const bool c_scr = c_scratch_wanted(C, ldc, 2, M, N);
    const int64_t ldc_p = (N + 7) / 8 * 8;
    const size_t bytes_c = c_scr ? pad256((size_t)M * ldc_p * 2) : 0;
    Scratch ws;
    const size_t total = bytes_a + bytes_b + bytes_w + bytes_n + bytes_c;
    if (total > 0) {
      e = ws.get(total, stream);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    char* wp = (char*)ws.ptr;
    float* sk_ws = (float*)(wp + bytes_a + bytes_b);
    unsigned int* sk_cnt = (unsigned int*)(wp + bytes_a + bytes_b + bytes_w);
    void* Cd = c_scr ? (void*)(wp + bytes_a + bytes_b + bytes_w + bytes_n) : C;
    const int64_t ldcd = c_scr ? ldc_p : ldc;
    if (c_scr && beta != 0.f) e = launch_repack_16(M, N, C, ldc, Cd, ldc_p, ctx);
    if (e == cudaSuccess && pl.cnt_bytes > 0)
      e = cudaMemsetAsync(sk_cnt, 0, pl.cnt_bytes, stream);
    const void* Ad = A;
    const void* Bd = B;
    int64_t ldad = lda, ldbd = ldb;
    if (e == cudaSuccess && !a_ok) {
      e = launch_repack_16((int)a_rows, (int)a_cols, A, lda, wp, lda_p, ctx);
      Ad = wp; ldad = lda_p;
    }
    if (e == cudaSuccess && !b_ok) {
      e = launch_repack_16((int)b_rows, (int)b_cols, B, ldb, wp + bytes_a, ldb_p, ctx);
      Bd = wp + bytes_a; ldbd = ldb_p;
    }
    if (e == cudaSuccess) {
      HgemmArgs a{transA, transB, M, N, K, Ad, ldad, Bd, ldbd, Cd, ldcd, alpha, beta, sms, bn,
                  c_tma_enabled(), g_fault_injection.load()};
      a.dtype = dtype;
      a.plan = pl;
      a.sk_ws = sk_ws;
      a.sk_cnt = sk_cnt;
      a.ep = ep;
      path = pl.sk_workers > 0 ? GEMM_PATH_TC_SPLITK : GEMM_PATH_TC;
      e = timed_hgemm(a, ctx);
      if (e == cudaSuccess && c_scr) e = launch_copy_rows(2, M, N, Cd, ldc_p, C, ldc, ctx);
    }
  }
  g_total_launches += ctx.launches;
  tl_last_grid = ctx.grid;
  if (e != cudaSuccess) {
    tl_last_path = GEMM_PATH_NONE;
    tl_last_launches = ctx.launches;
    return cuda_fail(e);
  }
  tl_last_path = path;
  tl_last_launches = ctx.launches;
  return GEMM_OK;
}

// gemm_host on large problems: row panels of C, so that the copies of later
// panels' A rows in and earlier panels' C rows out overlap the GEMMs.  One
// copy stream each way per device, created once; ordering by events.
cudaStream_t g_side[MAX_DEVICES][2];

cudaError_t side_streams(cudaStream_t* in, cudaStream_t* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  for (int i = 0; i < 2; ++i)
    if (!g_side[dev][i]) {
      e = cudaStreamCreateWithFlags(&g_side[dev][i], cudaStreamNonBlocking);
      if (e != cudaSuccess) return e;
    }
  *in = g_side[dev][0];
  *out = g_side[dev][1];
  return cudaSuccess;
}

struct EventSet {
  static constexpr int CAP = 2 * 72 + 2 + 16;
  cudaEvent_t ev[CAP] = {};
  int n = 0;
  ~EventSet() {
    for (int i = 0; i < n; ++i) cudaEventDestroy(ev[i]);
  }
  cudaError_t make(int count) {
    if (count > CAP) return cudaErrorInvalidValue;
    for (; n < count; ++n) {
      cudaError_t e = cudaEventCreateWithFlags(&ev[n], cudaEventDisableTiming);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
};

// gemm_host's pipeline events, kept per thread and device: created on first
// use and reused, since every call synchronises before it returns (no event
// is still pending when the next call records it).  Creating them per call
// put ~20 event creations ahead of the first copy.
EventSet* host_events(int dev) {
  thread_local std::unique_ptr<EventSet> sets[MAX_DEVICES];
  if (dev < 0 || dev >= MAX_DEVICES) return nullptr;
  if (!sets[dev]) sets[dev].reset(new EventSet());
  return sets[dev].get();
}

// Host buffers in, `panels` row panels of C computed and copied out as each
// finishes; returns after the caller's stream has synchronised.
int host_pipelined(int transA, int transB, int64_t M, int64_t N, int64_t K, int dtype,
                   float alpha, float beta, const void* A, int64_t lda, const void* B,
                   int64_t ldb, void* C, int64_t ldc, cudaStream_t stream, int64_t ar,
                   int64_t ac, int64_t br, int64_t bc, int panels) {
  const int64_t e = esize(dtype);
  const int64_t align = 16 / e;
  const int64_t lda_d = (ac + align - 1) / align * align;
  const int64_t ldb_d = (bc + align - 1) / align * align;
  const int64_t ldc_d = (N + align - 1) / align * align;
  const size_t nA = (size_t)(ar * lda_d * e + 255) / 256 * 256;
  const size_t nB = (size_t)(br * ldb_d * e + 255) / 256 * 256;
  const size_t nC = (size_t)(M * ldc_d * e + 255) / 256 * 256;
  // fp32 C: the first panel runs as NK products over K slices, each started
  // once its slice of B (and of the panel's A rows) has arrived, accumulating
  // in C (beta = 1 after the first); so the first GEMM waits for a quarter of
  // B rather than all of it.  (16-bit C would be rounded between slices.)
  const HostSched hs = host_sched_env();
  if (hs.panels > 0) panels = hs.panels < 64 ? hs.panels : 64;
  int NK = is_f32(dtype) && K >= 1024 ? 4 : 1;
  if (hs.kslices > 0 && is_f32(dtype)) NK = hs.kslices < 16 ? hs.kslices : 16;
  // (measured at 4096^3 fp32, whole calls: the last panel in two pieces
  // 2.353 ms, in one 2.37-2.38, in four 2.37; 8 panels 2.40-2.44; 2 K slices
  // 2.38, 8 K slices 2.47)
  const int tail = hs.tail > 0 ? (hs.tail < 8 ? hs.tail : 8) : 2;
  const int64_t kl = ((K + NK - 1) / NK + 63) / 64 * 64;  // K per slice
  // row ranges: panels of a whole number of 128-row tiles, the last one cut
  // into `tail` pieces
  int64_t rows[72];
  int np = 0;
  {
    const int64_t pr = ((M + panels - 1) / panels + 127) / 128 * 128;
    int64_t r = 0;
    for (int p = 0; p < panels - 1 && r < M && np < 64; ++p, r += pr) rows[np++] = r;
    if (r < M) {
      const int64_t left = M - r;
      const int64_t tr = ((left + tail - 1) / tail + 127) / 128 * 128;
      for (int t = 0; t < tail && r < M && np < 71; ++t, r += tr) rows[np++] = r;
    }
    rows[np] = M;
  }
  cudaStream_t sin, sout;
  cudaError_t ce = side_streams(&sin, &sout);
  if (ce != cudaSuccess) return cuda_fail(ce);
  int dev = 0;
  ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return cuda_fail(ce);
  EventSet* evp = host_events(dev);
  if (!evp) return GEMM_ERR_UNSUPPORTED;
  EventSet& evs = *evp;
  ce = evs.make(2 * np + 2 + NK);
  if (ce != cudaSuccess) return cuda_fail(ce);
  Scratch buf;
  ce = buf.get(nA + nB + nC, stream);
  if (ce != cudaSuccess) return cuda_fail(ce);
  char* dA = (char*)buf.ptr;
  char* dB = dA + nA;
  char* dC = dB + nB;
  cudaEvent_t ev_alloc = evs.ev[2 * np], ev_out = evs.ev[2 * np + 1];
  int path = GEMM_PATH_NONE, launches = 0;
  ce = cudaEventRecord(ev_alloc, stream);
  if (ce == cudaSuccess) ce = cudaStreamWaitEvent(sin, ev_alloc, 0);
  if (ce == cudaSuccess) ce = cudaStreamWaitEvent(sout, ev_alloc, 0);
  if (ce == cudaSuccess && NK == 1)
    ce = cudaMemcpy2DAsync(dB, ldb_d * e, B, ldb * e, bc * e, br, cudaMemcpyHostToDevice, sin);
  int rc = GEMM_OK;
  for (int p = 0; p < np && ce == cudaSuccess && rc == GEMM_OK; ++p) {
    const int64_t r0 = rows[p], r1 = rows[p + 1];
    const int64_t mp = r1 - r0;
    if (p == 0 && NK > 1) {
      // panel 0 (rows 0 .. mp), slice by slice: B rows k0..k1 of B[K,N] or
      // columns of B[N,K]; A columns k0..k1 of A[M,K] or rows of A[K,M]
      char* dC0 = dC;
      char* hC0 = static_cast<char*>(C);
      for (int c = 0; c < NK && ce == cudaSuccess && rc == GEMM_OK; ++c) {
        const int64_t k0 = c * kl, k1 = k0 + kl < K ? k0 + kl : K;
        if (k0 >= K) break;
        const int64_t kw = k1 - k0;
        const char* hB = static_cast<const char*>(B) + (transB ? k0 * e : k0 * ldb * e);
        char* dBk = dB + (transB ? k0 * e : k0 * ldb_d * e);
        ce = transB ? cudaMemcpy2DAsync(dBk, ldb_d * e, hB, ldb * e, kw * e, br,
                                        cudaMemcpyHostToDevice, sin)
                    : cudaMemcpy2DAsync(dBk, ldb_d * e, hB, ldb * e, bc * e, kw,
                                        cudaMemcpyHostToDevice, sin);
        const char* hA = static_cast<const char*>(A) + (transA ? k0 * lda * e : k0 * e);
        char* dAk = dA + (transA ? k0 * lda_d * e : k0 * e);
        if (ce == cudaSuccess)
          ce = transA ? cudaMemcpy2DAsync(dAk, lda_d * e, hA, lda * e, mp * e, kw,
                                          cudaMemcpyHostToDevice, sin)
                      : cudaMemcpy2DAsync(dAk, lda_d * e, hA, lda * e, kw * e, mp,
                                          cudaMemcpyHostToDevice, sin);
        if (ce == cudaSuccess && c == 0 && beta != 0.f)
          ce = cudaMemcpy2DAsync(dC0, ldc_d * e, hC0, ldc * e, N * e, mp, cudaMemcpyHostToDevice,
                                 sin);
        cudaEvent_t evk = evs.ev[2 * np + 2 + c];
        if (ce == cudaSuccess) ce = cudaEventRecord(evk, sin);
        if (ce == cudaSuccess) ce = cudaStreamWaitEvent(stream, evk, 0);
        if (ce != cudaSuccess) break;
        rc = run_gemm(transA, transB, mp, N, kw, dtype, alpha, c == 0 ? beta : 1.f, dAk, lda_d,
                      dBk, ldb_d, dC0, ldc_d, stream, transA ? kw : mp, transA ? mp : kw,
                      transB ? N : kw, transB ? kw : N);
        if (rc != GEMM_OK) break;
        path = tl_last_path;
        launches += tl_last_launches;
      }
      if (ce != cudaSuccess || rc != GEMM_OK) break;
      ce = cudaEventRecord(evs.ev[1], stream);
      if (ce == cudaSuccess) ce = cudaStreamWaitEvent(sout, evs.ev[1], 0);
      if (ce == cudaSuccess)
        ce = cudaMemcpy2DAsync(hC0, ldc * e, dC0, ldc_d * e, N * e, mp, cudaMemcpyDeviceToHost,
                               sout);
      continue;
    }
    // A rows r0..r1 of op(A): rows of A[M,K], or columns of A[K,M]
    const char* srcA = static_cast<const char*>(A) + (transA ? r0 * e : r0 * lda * e);
    char* dstA = dA + (transA ? r0 * e : r0 * lda_d * e);
    ce = transA ? cudaMemcpy2DAsync(dstA, lda_d * e, srcA, lda * e, mp * e, ar,
                                    cudaMemcpyHostToDevice, sin)
                : cudaMemcpy2DAsync(dstA, lda_d * e, srcA, lda * e, ac * e, mp,
                                    cudaMemcpyHostToDevice, sin);
    char* dCp = dC + r0 * ldc_d * e;
    char* hCp = static_cast<char*>(C) + r0 * ldc * e;
    if (ce == cudaSuccess && beta != 0.f)
      ce = cudaMemcpy2DAsync(dCp, ldc_d * e, hCp, ldc * e, N * e, mp, cudaMemcpyHostToDevice, sin);
    if (ce == cudaSuccess) ce = cudaEventRecord(evs.ev[2 * p], sin);
    if (ce == cudaSuccess) ce = cudaStreamWaitEvent(stream, evs.ev[2 * p], 0);
    if (ce != cudaSuccess) break;
    rc = run_gemm(transA, transB, mp, N, K, dtype, alpha, beta, dstA, lda_d, dB, ldb_d, dCp,
                  ldc_d, stream, transA ? K : mp, transA ? mp : K, br, bc);
    if (rc != GEMM_OK) break;
    path = tl_last_path;
    launches += tl_last_launches;
    ce = cudaEventRecord(evs.ev[2 * p + 1], stream);
    if (ce == cudaSuccess) ce = cudaStreamWaitEvent(sout, evs.ev[2 * p + 1], 0);
    if (ce == cudaSuccess)
      ce = cudaMemcpy2DAsync(hCp, ldc * e, dCp, ldc_d * e, N * e, mp, cudaMemcpyDeviceToHost,
                             sout);
  }
  // the caller's stream takes over both copy streams' work before the buffer
  // is released on it
  cudaError_t ce2 = cudaEventRecord(ev_out, sout);
  if (ce2 == cudaSuccess) ce2 = cudaStreamWaitEvent(stream, ev_out, 0);
  cudaError_t ce3 = cudaEventRecord(ev_alloc, sin);
  if (ce3 == cudaSuccess) ce3 = cudaStreamWaitEvent(stream, ev_alloc, 0);
  cudaFreeAsync(buf.ptr, stream);
  buf.ptr = nullptr;
  cudaError_t ce4 = cudaStreamSynchronize(stream);
  if (rc != GEMM_OK) return rc;
  if (ce != cudaSuccess) return cuda_fail(ce);
  if (ce2 != cudaSuccess || ce3 != cudaSuccess || ce4 != cudaSuccess) return GEMM_ERR_CUDA;
  tl_last_path = path;
  tl_last_launches = launches;
  return GEMM_OK;
}

// Strided batch (gemm_strided_batched): one launch over the whole batch when
// the operands allow it, else entry by entry through run_gemm.  Arguments
// already checked; batch >= 2, M, N > 0.
int run_batched(int transA, int transB, int64_t M64, int64_t N64, int64_t K64, int dtype,
                float alpha, float beta, const void* A, int64_t lda, int64_t sA, const void* B,
                int64_t ldb, int64_t sB, void* C, int64_t ldc, int64_t sC, int64_t batch,
                cudaStream_t stream, int64_t a_rows, int64_t a_cols, int64_t b_rows,
                int64_t b_cols) {
  int dev, sms;
  unsigned int* status;
  int rc = device_state(&dev, &status, &sms);
  if (rc != GEMM_OK) return rc;
  const int M = (int)M64, N = (int)N64, K = (int)K64;
  const int64_t es = esize(dtype);
  const char* Ab = static_cast<const char*>(A);
  const char* Bb = static_cast<const char*>(B);
  char* Cb = static_cast<char*>(C);
  // (TF32 runs entry by entry: its operands may need packing into K-major rows)
  const bool tma_ok = !is_f32(dtype) && ((uintptr_t)A % 16) == 0 &&
                      ((uintptr_t)B % 16) == 0 &&
                      (lda % 8) == 0 && (ldb % 8) == 0 && (sA % 8) == 0 && (sB % 8) == 0;
  LaunchCtx ctx{stream, status, (uint64_t)g_timeout_ns.load(), 0};
  int path = GEMM_PATH_NONE;
  cudaError_t e = cudaSuccess;
  bool per_entry = K > 0 && dtype != GEMM_F32 && !tma_ok;
  if (!per_entry && K > 0 && dtype != GEMM_F32) {
    // one persistent launch walks (entry, tile) units; the unit count stays
    // below 2^31 by cutting very large batches into groups
    path = GEMM_PATH_TC_BATCHED;
    const int64_t tiles = (int64_t)((M + HG_BM - 1) / HG_BM) * ((N + 31) / 32);
    const int64_t per_launch = tiles > 0 ? (int64_t)0x7fffffff / tiles : batch;
    for (int64_t b0 = 0; b0 < batch && e == cudaSuccess; b0 += per_launch) {
      const int nb = (int)(batch - b0 < per_launch ? batch - b0 : per_launch);
      const int bn = pick_bn16(M, N, K, transA, transB, sms, nb, 0);
      HgemmArgs a{transA, transB, M, N, K, Ab + b0 * sA * es, lda, Bb + b0 * sB * es, ldb,
                  Cb + b0 * sC * es, ldc, alpha, beta, sms, bn, c_tma_enabled(),
                  g_fault_injection.load()};
      a.dtype = dtype;
      a.batch = nb;
      // whole tiles: the batch itself fills the grid
      a.plan = hgemm_plan(M, N, K, bn, transA, transB, HG_BK, nb, pair_enabled(), sms, 0);
      a.stride_a = sA; a.stride_b = sB; a.stride_c = sC;
      e = timed_hgemm(a, ctx);
      // the driver refused the 3-D description (e.g. batch pitches that
      // interleave rows) before the first launch: run entry by entry
      if (e == cudaErrorNotSupported && ctx.launches == 0) {
        per_entry = true;
        e = cudaSuccess;
        break;
      }
    }
  }
  if (per_entry) {
    // entry by entry: each one is a full gemm() (padded copies included)
    int64_t launches = 0;
    for (int64_t b = 0; b < batch; ++b) {
      rc = run_gemm(transA, transB, M64, N64, K64, dtype, alpha, beta, Ab + b * sA * es, lda,
                    Bb + b * sB * es, ldb, Cb + b * sC * es, ldc, stream, a_rows, a_cols, b_rows,
                    b_cols);
      launches += tl_last_launches;
      if (rc != GEMM_OK) {
        tl_last_launches = (int)launches;
        return rc;
      }
    }
    tl_last_path = GEMM_PATH_PER_ENTRY;
    tl_last_launches = (int)launches;
    return GEMM_OK;
  }
  if (path == GEMM_PATH_TC_BATCHED) {
    // launched above
  } else if (K == 0) {
    path = GEMM_PATH_SCALE;
    for (int64_t b = 0; b < batch && e == cudaSuccess; ++b)
      e = launch_scale(out_kind(dtype), M, N, Cb + b * sC * es, ldc, beta, ctx);
  } else if (dtype == GEMM_F32) {
    // the batch runs on grid.y, at most 65535 entries per launch
    path = GEMM_PATH_FFMA_BATCHED;
    for (int64_t b0 = 0; b0 < batch && e == cudaSuccess; b0 += 65535) {
      const int nb = (int)(batch - b0 < 65535 ? batch - b0 : 65535);
      SgemmArgs a{transA, transB, M, N, K, (const float*)(Ab + b0 * sA * es), lda,
                  (const float*)(Bb + b0 * sB * es), ldb, (float*)(Cb + b0 * sC * es), ldc,
                  alpha, beta, 1, K, nullptr};
      a.batch = nb;
      a.stride_a = sA; a.stride_b = sB; a.stride_c = sC;
      e = timed_sgemm(a, ctx);
    }
  }
  g_total_launches += ctx.launches;
  tl_last_grid = ctx.grid;
  tl_last_launches = ctx.launches;
  if (e != cudaSuccess) {
    tl_last_path = GEMM_PATH_NONE;
    return cuda_fail(e);
  }
  tl_last_path = path;
  return GEMM_OK;
}

}  // namespace

extern "C" {

int gemm_strided_batched(int transA, int transB, int64_t M, int64_t N, int64_t K, int dtype,
                         float alpha, float beta, const void* A, int64_t lda, int64_t sA,
                         const void* B, int64_t ldb, int64_t sB, void* C, int64_t ldc,
                         int64_t sC, int64_t batch, gemm_stream_t stream) {
  int64_t ar, ac, br, bc;
  tl_last_path = GEMM_PATH_NONE;
  tl_last_launches = 0;
  if (batch < 0 || sA < 0 || sB < 0 || sC < 0) return GEMM_ERR_INVALID_ARG;
  int rc = check_args(transA, transB, M, N, K, dtype, A, lda, B, ldb, C, ldc, &ar, &ac, &br, &bc);
  if (rc != GEMM_OK) return rc;
  if (batch == 0 || M == 0 || N == 0) return GEMM_OK;
  if (batch >= ((int64_t)1 << 31)) return GEMM_ERR_UNSUPPORTED;
  if (batch == 1)
    return run_gemm(transA, transB, M, N, K, dtype, alpha, beta, A, lda, B, ldb, C, ldc,
                    (cudaStream_t)stream, ar, ac, br, bc);
  const int64_t es = esize(dtype);
  const int64_t fc = footprint_bytes(M, N, ldc, 1);  // elements of one C
  if (sC < fc) return GEMM_ERR_ALIAS;                 // C entries would overlap
  // whole extents, in bytes, without overflow
  const int64_t big = (int64_t)1 << 62;
  auto span = [&](int64_t foot, int64_t stride, int64_t* out) {
    if (stride > 0 && (batch - 1) > (big / es - foot) / stride) return false;
    *out = ((batch - 1) * stride + foot) * es;
    return true;
  };
  int64_t nC = 0, nA = 0, nB = 0;
  if (!span(fc, sC, &nC)) return GEMM_ERR_UNSUPPORTED;
  if (K > 0) {
    if (!span(footprint_bytes(ar, ac, lda, 1), sA, &nA) ||
        !span(footprint_bytes(br, bc, ldb, 1), sB, &nB))
      return GEMM_ERR_UNSUPPORTED;
    if (overlaps(C, nC, A, nA) || overlaps(C, nC, B, nB)) return GEMM_ERR_ALIAS;
  }
  return run_batched(transA, transB, M, N, K, dtype, alpha, beta, A, lda, sA, B, ldb, sB, C, ldc,
                     sC, batch, (cudaStream_t)stream, ar, ac, br, bc);
}

int gemm_ex(int transA, int transB, int64_t M, int64_t N, int64_t K, int dtype, float alpha,
            float beta, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
            int64_t ldc, const void* bias, int act, gemm_stream_t stream) {
  int64_t ar, ac, br, bc;
  tl_last_path = GEMM_PATH_NONE;
  tl_last_launches = 0;
  if (act != GEMM_ACT_NONE && act != GEMM_ACT_RELU && act != GEMM_ACT_GELU)
    return GEMM_ERR_INVALID_ARG;
  int rc = check_args(transA, transB, M, N, K, dtype, A, lda, B, ldb, C, ldc, &ar, &ac, &br, &bc);
  if (rc != GEMM_OK) return rc;
  if (M == 0 || N == 0) return GEMM_OK;
  const int64_t e = esize(dtype);
  if (bias) {
    if (((uintptr_t)bias % (uintptr_t)e) != 0) return GEMM_ERR_INVALID_ARG;
    if (overlaps(C, footprint_bytes(M, N, ldc, e), bias, N * e)) return GEMM_ERR_ALIAS;
  }
  Epilogue ep;
  ep.bias = bias;
  ep.act = act;
  return run_gemm(transA, transB, M, N, K, dtype, alpha, beta, A, lda, B, ldb, C, ldc,
                  (cudaStream_t)stream, ar, ac, br, bc, ep);
}

int gemm(int transA, int transB, int64_t M, int64_t N, int64_t K, int dtype, float alpha,
         float beta, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
         int64_t ldc, gemm_stream_t stream) {
  int64_t ar, ac, br, bc;
  tl_last_path = GEMM_PATH_NONE;
  tl_last_launches = 0;
  int rc = check_args(transA, transB, M, N, K, dtype, A, lda, B, ldb, C, ldc, &ar, &ac, &br, &bc);
  if (rc != GEMM_OK) return rc;
  if (M == 0 || N == 0) return GEMM_OK;
  return run_gemm(transA, transB, M, N, K, dtype, alpha, beta, A, lda, B, ldb, C, ldc,
                  (cudaStream_t)stream, ar, ac, br, bc);
}

int gemm_host(int transA, int transB, int64_t M, int64_t N, int64_t K, int dtype, float alpha,
              float beta, const void* A, int64_t lda, const void* B, int64_t ldb, void* C,
              int64_t ldc, gemm_stream_t stream_) {
  int64_t ar, ac, br, bc;
  tl_last_path = GEMM_PATH_NONE;
  tl_last_launches = 0;
  int rc = check_args(transA, transB, M, N, K, dtype, A, lda, B, ldb, C, ldc, &ar, &ac, &br, &bc);
  if (rc != GEMM_OK) return rc;
  if (M == 0 || N == 0) return GEMM_OK;
  cudaStream_t stream = (cudaStream_t)stream_;
  // large problems: copies overlapped with the GEMMs of row panels
  if (K > 0 && M >= 256 && (double)M * N * K >= (double)(1ll << 30) && host_pipeline_enabled())
    return host_pipelined(transA, transB, M, N, K, dtype, alpha, beta, A, lda, B, ldb, C, ldc,
                          stream, ar, ac, br, bc, M >= 4096 ? 4 : 2);
  const int64_t e = esize(dtype);
  const int64_t align = 16 / e;  // device pitch: whole 16-byte units
  const int64_t lda_d = (ac + align - 1) / align * align;
  const int64_t ldb_d = (bc + align - 1) / align * align;
  const int64_t ldc_d = (N + align - 1) / align * align;
  const size_t nA = K > 0 ? (size_t)(ar * lda_d * e + 255) / 256 * 256 : 0;
  const size_t nB = K > 0 ? (size_t)(br * ldb_d * e + 255) / 256 * 256 : 0;
  const size_t nC = (size_t)(M * ldc_d * e + 255) / 256 * 256;
  Scratch buf;
  cudaError_t ce = buf.get(nA + nB + nC, stream);
  if (ce != cudaSuccess) return cuda_fail(ce);
  char* dA = (char*)buf.ptr;
  char* dB = dA + nA;
  char* dC = dB + nB;
  if (K > 0) {
    ce = cudaMemcpy2DAsync(dA, lda_d * e, A, lda * e, ac * e, ar, cudaMemcpyHostToDevice, stream);
    if (ce == cudaSuccess)
      ce = cudaMemcpy2DAsync(dB, ldb_d * e, B, ldb * e, bc * e, br, cudaMemcpyHostToDevice,
                             stream);
  }
  if (ce == cudaSuccess && beta != 0.f)
    ce = cudaMemcpy2DAsync(dC, ldc_d * e, C, ldc * e, N * e, M, cudaMemcpyHostToDevice, stream);
  if (ce != cudaSuccess) return cuda_fail(ce);
  rc = run_gemm(transA, transB, M, N, K, dtype, alpha, beta, dA, lda_d, dB, ldb_d, dC, ldc_d,
                stream, ar, ac, br, bc);
  if (rc != GEMM_OK) return rc;
  const int path = tl_last_path, launches = tl_last_launches;
  ce = cudaMemcpy2DAsync(C, ldc * e, dC, ldc_d * e, N * e, M, cudaMemcpyDeviceToHost, stream);
  if (ce != cudaSuccess) return cuda_fail(ce);
  cudaFreeAsync(buf.ptr, stream);
  buf.ptr = nullptr;
  ce = cudaStreamSynchronize(stream);
  tl_last_path = path;
  tl_last_launches = launches;
  return ce == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}

int gemm_check_device_status(gemm_stream_t stream) {
  int dev, sms;
  unsigned int* status;
  int rc = device_state(&dev, &status, &sms);
  if (rc != GEMM_OK) return rc;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return GEMM_ERR_CUDA;
  unsigned int word = 0;
  if (cudaMemcpy(&word, status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return GEMM_ERR_CUDA;
  if (word != 0) {
    const unsigned int zero = 0;
    if (cudaMemcpy(status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return GEMM_ERR_CUDA;
    return GEMM_ERR_TIMEOUT;
  }
  return GEMM_OK;
}

const char* gemm_status_string(int status) {
  switch (status) {
    case GEMM_OK: return "GEMM_OK";
    case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG";
    case GEMM_ERR_UNSUPPORTED: return "GEMM_ERR_UNSUPPORTED";
    case GEMM_ERR_ALIAS: return "GEMM_ERR_ALIAS";
    case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA";
    case GEMM_ERR_NO_MEMORY: return "GEMM_ERR_NO_MEMORY";
    case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT";
    default: return "GEMM_ERR_UNKNOWN";
  }
}

int gemm_version(void) { return (1 << 16) | 0; }

int64_t gemm_scratch_high_water(int reset) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return -1;
  cudaMemPool_t pool;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    pool = g_pool[dev];
  }
  if (!pool) return 0;
  cuuint64_t v = 0;
  if (cudaMemPoolGetAttribute(pool, cudaMemPoolAttrUsedMemHigh, &v) != cudaSuccess) return -1;
  if (reset) {
    cuuint64_t zero = 0;
    if (cudaMemPoolSetAttribute(pool, cudaMemPoolAttrUsedMemHigh, &zero) != cudaSuccess)
      return -1;
  }
  return (int64_t)v;
}

int gemm_last_path(void) { return tl_last_path; }
int gemm_last_launches(void) { return tl_last_launches; }
int gemm_last_grid(void) { return tl_last_grid; }
int64_t gemm_total_launches(void) { return g_total_launches.load(); }

void gemm_set_wait_timeout_ns(int64_t ns) {
  g_timeout_ns.store(ns > 0 ? ns : 2000000000LL);
}

void gemm_set_fault_injection(int mode) { g_fault_injection.store(mode); }

void gemm_set_kernel_events(void* start, void* end) {
  tl_ev_start = (start && end) ? static_cast<cudaEvent_t>(start) : nullptr;
  tl_ev_end = (start && end) ? static_cast<cudaEvent_t>(end) : nullptr;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// gemm_splitk_noalloc: the same product for callers that must not allocate
// device memory, e.g. code running under an allocator that already owns the
// whole device (a framework's caching allocator), or a host process whose
// rules forbid runtime allocation once it is serving.  The partial sums that
// gemm() keeps in memory from the stream-ordered allocator (the fp32 kernel's
// K slices; the tensor-core kernel's shared tiles and their arrival counters)
// live here in a fixed array compiled into the library instead.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds it (GEMM_NOALLOC_SCRATCH_BYTES) until the process exits.  Host
// code cannot use its name as a device address, so its address is looked up
// once per device with cudaGetSymbolAddress, with that device current, the
// first time the entry point runs on it; that first call therefore makes a
// runtime query and should come before any stream capture.  All calls share
// the one array and it keeps whatever the last call left: every partial sum a
// call reads is written by the same call first, and the arrival counters,
// which must start at zero, are cleared on the stream (cudaMemsetAsync, no
// allocation) before each launch that uses them; two calls that overlap on
// the GPU (different streams, no ordering between them) race on it.
// ---------------------------------------------------------------------------
#define GEMM_NOALLOC_SCRATCH_BYTES (8u << 20)

static __device__ __align__(256) float g_noalloc_scratch[GEMM_NOALLOC_SCRATCH_BYTES / sizeof(float)];

namespace {
float* g_noalloc_ptr[MAX_DEVICES];

int noalloc_scratch(int dev, float** out) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return GEMM_ERR_CUDA;
    g_noalloc_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return GEMM_OK;
}
}  // namespace

extern "C" int gemm_splitk_noalloc(int transA, int transB, int64_t M, int64_t N, int64_t K,
                                   int dtype, float alpha, float beta, const void* A,
                                   int64_t lda, const void* B, int64_t ldb, void* C,
                                   int64_t ldc, gemm_stream_t stream_) {
  int64_t ar, ac, br, bc;
  tl_last_path = GEMM_PATH_NONE;
  tl_last_launches = 0;
  int rc = check_args(transA, transB, M, N, K, dtype, A, lda, B, ldb, C, ldc, &ar, &ac, &br, &bc);
  if (rc != GEMM_OK) return rc;
  if (dtype == GEMM_F32_TF32 || dtype == GEMM_F32_3XTF32)
    return GEMM_ERR_UNSUPPORTED;  // their packing would need scratch
  if (M == 0 || N == 0) return GEMM_OK;
  cudaStream_t stream = (cudaStream_t)stream_;
  int dev, sms;
  unsigned int* status;
  rc = device_state(&dev, &status, &sms);
  if (rc != GEMM_OK) return rc;
  float* scratch = nullptr;
  rc = noalloc_scratch(dev, &scratch);
  if (rc != GEMM_OK) return rc;
  LaunchCtx ctx{stream, status, (uint64_t)g_timeout_ns.load(), 0};
  const int Mi = (int)M, Ni = (int)N, Ki = (int)K;
  int path = GEMM_PATH_NONE;
  cudaError_t e = cudaSuccess;
  if (Ki == 0) {
    path = GEMM_PATH_SCALE;
    e = launch_scale(dtype, Mi, Ni, C, ldc, beta, ctx);
  } else if (dtype == GEMM_F32) {
    // gemm()'s tile and K split; without gemm()'s operand packing and
    // stream-K launch on large problems, which take scratch
    int tile, splits, k_slice;
    int64_t tiles;
    plan_f32(Mi, Ni, Ki, sms, &tile, &tiles, &splits, &k_slice);
    if (splits > 1 && (uint64_t)splits * (uint64_t)M * (uint64_t)N * sizeof(float) >
                          GEMM_NOALLOC_SCRATCH_BYTES)
      return GEMM_ERR_UNSUPPORTED;  // partial sums would not fit the fixed array
    SgemmArgs a{transA, transB, Mi, Ni, Ki, (const float*)A, lda, (const float*)B, ldb,
                (float*)C, ldc, alpha, beta, splits, k_slice, splits > 1 ? scratch : nullptr};
    a.tile = tile;
    path = splits > 1 ? GEMM_PATH_FFMA_SPLITK : GEMM_PATH_FFMA;
    e = timed_sgemm(a, ctx);
    if (e == cudaSuccess && splits > 1)
      e = launch_splitk_reduce(0, Mi, Ni, splits, scratch, C, ldc, alpha, beta, ctx);
  } else {
    // fp16 operands must already meet the tensor-memory-access unit's rules
    // (16-byte aligned base and row pitch): padding them would need scratch.
    if (((uintptr_t)A % 16) != 0 || (lda % 8) != 0 || ((uintptr_t)B % 16) != 0 || (ldb % 8) != 0)
      return GEMM_ERR_UNSUPPORTED;
    // gemm()'s tile width and schedule; shared tiles' partial sums and
    // counters in the fixed array when they fit, else whole tiles only
    const int bn = pick_bn16(Mi, Ni, Ki, transA, transB, sms, 1, sk_mode());
    HPlan pl = hgemm_plan(Mi, Ni, Ki, bn, transA, transB, HG_BK, 1, pair_enabled(), sms,
                          sk_mode());
    if (pad256(pl.ws_bytes) + pl.cnt_bytes > GEMM_NOALLOC_SCRATCH_BYTES)
      pl = hgemm_plan(Mi, Ni, Ki, bn, transA, transB, HG_BK, 1, pair_enabled(), sms, 0);
    unsigned int* cnt = reinterpret_cast<unsigned int*>(
        reinterpret_cast<char*>(scratch) + pad256(pl.ws_bytes));
    if (pl.cnt_bytes > 0) e = cudaMemsetAsync(cnt, 0, pl.cnt_bytes, stream);
    HgemmArgs a{transA, transB, Mi, Ni, Ki, A, lda, B, ldb, C, ldc, alpha, beta, sms, bn,
                c_tma_enabled(), g_fault_injection.load()};
    a.dtype = dtype;
    a.plan = pl;
    a.sk_ws = scratch;
    a.sk_cnt = cnt;
    path = pl.sk_workers > 0 ? GEMM_PATH_TC_SPLITK : GEMM_PATH_TC;
    if (e == cudaSuccess) e = timed_hgemm(a, ctx);
  }
  g_total_launches += ctx.launches;
  tl_last_launches = ctx.launches;
  tl_last_grid = ctx.grid;
  if (e != cudaSuccess) return cuda_fail(e);
  tl_last_path = path;
  return GEMM_OK;
}
