// Small memory-bound kernels around the GEMM main loops.
//
//  splitk_reduce : C = alpha * sum_z P[z] + beta * C, the reduction step of
//                  split-K ("Metal GEMM Kernels for LoRA Training", section 5:
//                  the K range is cut into chunks, each chunk writes fp32 partial
//                  sums to device memory, a second pass adds them).  The slices
//                  are added in increasing z, so the result does not depend on
//                  scheduling.
//  scale         : C = beta * C, the K == 0 case of C = alpha*A*B + beta*C.
//  repack        : copies an operand whose rows are not 16-byte aligned into a
//                  zero-padded buffer with a 16-byte row pitch, so that the
//                  tensor-memory-access unit (16-bit) or 16-byte copies (fp32)
//                  can read it.
//  copy_rows     : the way back: C computed into an aligned scratch copy is
//                  copied into the caller's unaligned rows.
//  transpose_f32 : packs an fp32 operand stored with k contiguous into the
//                  k-major layout the FP32 kernel reads fastest (the "packing"
//                  step of a tuned BLAS, "From a C loop to a GPU kernel", "What
//                  BLAS is buying").
//
// All are HBM-bound; they use grid-stride loops over 128-bit accesses
// where the layout allows, with grids sized to a multiple of the SM count.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "internal.h"

namespace gb300 {
namespace {

int sm_count() {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
  }
  return sms;
}

int grid_for(int64_t work_items, int threads) {
  int64_t blocks = (work_items + threads - 1) / threads;
  const int64_t cap = (int64_t)sm_count() * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return (int)blocks;
}

__device__ __forceinline__ void store_out(float* C, int64_t i, float v) { C[i] = v; }
__device__ __forceinline__ void store_out(__half* C, int64_t i, float v) {
  C[i] = __float2half_rn(v);
}
__device__ __forceinline__ float load_out(const float* C, int64_t i) { return C[i]; }
__device__ __forceinline__ float load_out(const __half* C, int64_t i) {
  return __half2float(C[i]);
}
__device__ __forceinline__ void store_out(__nv_bfloat16* C, int64_t i, float v) {
  C[i] = __float2bfloat16_rn(v);
}
__device__ __forceinline__ float load_out(const __nv_bfloat16* C, int64_t i) {
  return __bfloat162float(C[i]);
}

// One thread per 4 consecutive columns of a row (N % 4 == 0 path reads P with
// float4); the general path handles one element per thread.
template <typename T>
__global__ void splitk_reduce_vec4(int M, int N, int splits, const float* __restrict__ P, T* C,
                                   int64_t ldc, float alpha, float beta, Epilogue ep) {
  pdl_wait();
  pdl_trigger();
  const int64_t quads = (int64_t)M * (N / 4);
  const int64_t slice = (int64_t)M * N;
  for (int64_t q = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; q < quads;
       q += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = q / (N / 4);
    const int64_t n = (q - m * (N / 4)) * 4;
    const float* src = P + m * N + n;
    float4 s = *reinterpret_cast<const float4*>(src);
    for (int z = 1; z < splits; ++z) {
      const float4 t = *reinterpret_cast<const float4*>(src + z * slice);
      s.x += t.x; s.y += t.y; s.z += t.z; s.w += t.w;
    }
    const float v[4] = {s.x, s.y, s.z, s.w};
    const int64_t base = m * ldc + n;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float o = alpha * v[j];
      if (beta != 0.f) o = __fmaf_rn(beta, load_out(C, base + j), o);
      store_out(C, base + j, apply_epilogue<T>(o, ep, (int)n + j));
    }
  }
}

template <typename T>
__global__ void splitk_reduce_scalar(int M, int N, int splits, const float* __restrict__ P, T* C,
                                     int64_t ldc, float alpha, float beta, Epilogue ep) {
  pdl_wait();
  pdl_trigger();
  const int64_t total = (int64_t)M * N;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = i / N, n = i - m * N;
    float s = P[i];
    for (int z = 1; z < splits; ++z) s += P[i + z * total];
    float o = alpha * s;
    if (beta != 0.f) o = __fmaf_rn(beta, load_out(C, m * ldc + n), o);
    store_out(C, m * ldc + n, apply_epilogue<T>(o, ep, (int)n));
  }
}

template <typename T>
__global__ void scale_kernel(int M, int N, T* C, int64_t ldc, float beta, Epilogue ep) {
  pdl_wait();
  pdl_trigger();
  const int64_t total = (int64_t)M * N;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = i / N, n = i - m * N;
    const int64_t off = m * ldc + n;
    const float o = beta != 0.f ? beta * load_out(C, off) : 0.f;
    store_out(C, off, apply_epilogue<T>(o, ep, (int)n));
  }
}

// Row pitch change: element bit patterns (fp16, bf16 or fp32 alike) copied
// from rows of any alignment into rows of ld_dst elements, ld_dst a multiple
// of one 16-byte chunk; a thread writes one chunk with a 128-bit store and
// reads its elements one by one (coalesced across the warp); zeros past cols.
// Blocks run over (chunk range, row) pairs: no per-element division.
template <typename W>
__global__ void __launch_bounds__(256) repack_kernel(int rows, int cols, const W* __restrict__ src,
                                                     int64_t ld_src, W* __restrict__ dst,
                                                     int64_t ld_dst) {
  pdl_wait();
  pdl_trigger();
  constexpr int V = 16 / sizeof(W);
  const int chunks = (int)(ld_dst / V);
  for (int r = blockIdx.y; r < rows; r += gridDim.y) {
    const W* s = src + (int64_t)r * ld_src;
    for (int q = blockIdx.x * blockDim.x + threadIdx.x; q < chunks; q += gridDim.x * blockDim.x) {
      const int c0 = q * V;
      uint32_t w[4];
      if constexpr (sizeof(W) == 4) {
#pragma unroll
        for (int e = 0; e < 4; ++e) w[e] = (c0 + e < cols) ? (uint32_t)__ldg(s + c0 + e) : 0u;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t lo = (c0 + 2 * e < cols) ? (uint32_t)__ldg(s + c0 + 2 * e) : 0u;
          const uint32_t hi = (c0 + 2 * e + 1 < cols) ? (uint32_t)__ldg(s + c0 + 2 * e + 1) : 0u;
          w[e] = lo | (hi << 16);
        }
      }
      *reinterpret_cast<uint4*>(dst + (int64_t)r * ld_dst + c0) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// Plain row copy for rows of any alignment: element-wise on both sides
// (coalesced across the warp), eight elements a thread in flight.
template <typename W>
__global__ void __launch_bounds__(256) copy_rows_kernel(int rows, int cols,
                                                        const W* __restrict__ src, int64_t ld_src,
                                                        W* __restrict__ dst, int64_t ld_dst) {
  pdl_wait();
  pdl_trigger();
  constexpr int U = 8;
  for (int r = blockIdx.y; r < rows; r += gridDim.y) {
    const W* s = src + (int64_t)r * ld_src;
    W* d = dst + (int64_t)r * ld_dst;
    for (int c0 = blockIdx.x * blockDim.x * U + threadIdx.x; c0 < cols;
         c0 += gridDim.x * blockDim.x * U) {
      W v[U];
#pragma unroll
      for (int e = 0; e < U; ++e) {
        const int c = c0 + e * (int)blockDim.x;
        v[e] = c < cols ? __ldg(s + c) : W(0);
      }
#pragma unroll
      for (int e = 0; e < U; ++e) {
        const int c = c0 + e * (int)blockDim.x;
        if (c < cols) d[c] = v[e];
      }
    }
  }
}

// dst[c][r] = src[r][c] for a rows x cols fp32 matrix: 64 x 64 tiles staged
// through shared memory (one padding column), 128-bit global loads and stores
// where rows are 16-byte aligned, scalar accesses at ragged edges.
template <bool VEC>
__global__ void __launch_bounds__(256) transpose_f32_kernel(int rows, int cols,
                                                            const float* __restrict__ src,
                                                            int64_t ld_src, float* __restrict__ dst,
                                                            int64_t ld_dst) {
  pdl_wait();
  pdl_trigger();
  __shared__ float tile[64][65];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;  // 16 float4 columns x 16 rows
  const int tiles_c = (cols + 63) / 64;
  const int64_t tiles = (int64_t)((rows + 63) / 64) * tiles_c;
  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
    const int r0 = (int)(t / tiles_c) * 64, c0 = (int)(t % tiles_c) * 64;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const int rr = ty + 16 * p, r = r0 + rr, c = c0 + 4 * tx;
      float v[4];
      if (VEC && r < rows && c + 3 < cols) {
        const float4 f = __ldg(reinterpret_cast<const float4*>(src + (int64_t)r * ld_src + c));
        v[0] = f.x; v[1] = f.y; v[2] = f.z; v[3] = f.w;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          v[e] = (r < rows && c + e < cols) ? src[(int64_t)r * ld_src + c + e] : 0.f;
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) tile[rr][4 * tx + e] = v[e];
    }
    __syncthreads();
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const int cc = ty + 16 * p, c = c0 + cc, r = r0 + 4 * tx;  // dst row c, columns r..r+3
      if (c >= cols) continue;
      const float v0 = tile[4 * tx][cc], v1 = tile[4 * tx + 1][cc], v2 = tile[4 * tx + 2][cc],
                  v3 = tile[4 * tx + 3][cc];
      float* d = dst + (int64_t)c * ld_dst + r;
      if (VEC && r + 3 < rows) {
        *reinterpret_cast<float4*>(d) = make_float4(v0, v1, v2, v3);
      } else {
        const float v[4] = {v0, v1, v2, v3};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (r + e < rows) d[e] = v[e];
      }
    }
    __syncthreads();
  }
}

template <typename W>
cudaError_t launch_repack(int rows, int cols, const void* src, int64_t ld_src, void* dst,
                          int64_t ld_dst, LaunchCtx& ctx) {
  constexpr int V = 16 / sizeof(W);
  if (ld_dst % V != 0 || ld_dst < cols || (reinterpret_cast<uintptr_t>(dst) & 15u) != 0)
    return cudaErrorInvalidValue;
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  const int64_t chunks = ld_dst / V;
  const int gx = (int)std::min<int64_t>((chunks + 255) / 256, 64);
  const int gy = (int)std::min<int64_t>(std::min<int64_t>(rows, 65535),
                                        std::max<int64_t>(1, (int64_t)sm_count() * 8 / gx));
  cudaError_t e = launch_kernel(repack_kernel<W>, dim3(gx, gy), dim3(256), 0, ctx.stream, 1, rows,
                                cols, static_cast<const W*>(src), ld_src, static_cast<W*>(dst),
                                ld_dst);
  if (e == cudaSuccess) ctx.launches++;
  return e;
}

}  // namespace

cudaError_t launch_copy_rows(int esize, int rows, int cols, const void* src, int64_t ld_src,
                             void* dst, int64_t ld_dst, LaunchCtx& ctx) {
  if (esize != 2 && esize != 4) return cudaErrorInvalidValue;
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  const int64_t per_block = 256 * 8;
  const int gx = (int)std::min<int64_t>((cols + per_block - 1) / per_block, 64);
  const int gy = (int)std::min<int64_t>(std::min<int64_t>(rows, 65535),
                                        std::max<int64_t>(1, (int64_t)sm_count() * 8 / gx));
  cudaError_t e =
      esize == 2
          ? launch_kernel(copy_rows_kernel<uint16_t>, dim3(gx, gy), dim3(256), 0, ctx.stream, 1,
                          rows, cols, static_cast<const uint16_t*>(src), ld_src,
                          static_cast<uint16_t*>(dst), ld_dst)
          : launch_kernel(copy_rows_kernel<uint32_t>, dim3(gx, gy), dim3(256), 0, ctx.stream, 1,
                          rows, cols, static_cast<const uint32_t*>(src), ld_src,
                          static_cast<uint32_t*>(dst), ld_dst);
  if (e == cudaSuccess) ctx.launches++;
  return e;
}

// ---------------------------------------------------------------- 3xTF32 split
// An fp32 value x as hi + lo with hi its TF32 part (sign, exponent and the
// top 10 fraction bits: x with the low 13 fraction bits cleared, i.e.
// truncated toward zero) and lo = x - hi, which is exact in fp32 (hi and x
// share their leading bits) and below 2^-10 |x|.  A tensor core fed hi and lo
// as TF32 operands recovers x * y, to about 2^-20 relative, as hi(x) hi(y) +
// hi(x) lo(y) + lo(x) hi(y).  Infinities and NaNs are kept in hi (lo = 0).
__device__ __forceinline__ void tf32_split(float x, float& hi, float& lo) {
  if (!isfinite(x)) {
    hi = x;
    lo = 0.f;
    return;
  }
  hi = __uint_as_float(__float_as_uint(x) & 0xffffe000u);
  lo = x - hi;
}

// dst_hi[r][c], dst_lo[r][c] (row pitch ld_dst, 16-byte aligned rows) from
// src[r][c] for c < cols, zero for cols <= c < ld_dst.  One thread per 4
// destination columns.
__global__ void __launch_bounds__(256) split_rows_kernel(int rows, int cols,
                                                         const float* __restrict__ src,
                                                         int64_t ld_src, float* __restrict__ hi,
                                                         float* __restrict__ lo, int64_t ld_dst) {
  pdl_wait();
  pdl_trigger();
  const int q = (int)(ld_dst / 4);
  const int64_t total = (int64_t)rows * q;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(i / q), c = (int)(i - (int64_t)r * q) * 4;
    float h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float x = c + e < cols ? src[(int64_t)r * ld_src + c + e] : 0.f;
      tf32_split(x, h[e], l[e]);
    }
    *reinterpret_cast<float4*>(hi + (int64_t)r * ld_dst + c) = make_float4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<float4*>(lo + (int64_t)r * ld_dst + c) = make_float4(l[0], l[1], l[2], l[3]);
  }
}

// The transposing counterpart: dst[c][r] from src[r][c] (src rows x cols,
// dst cols x rows), 64 x 64 tiles through shared memory as in
// transpose_f32_kernel, split on the way out.  Destination columns r in
// [rows, ld_dst) are not written (the caller zeroes them or never reads them).
__global__ void __launch_bounds__(256) split_transpose_kernel(int rows, int cols,
                                                              const float* __restrict__ src,
                                                              int64_t ld_src, float* __restrict__ hi,
                                                              float* __restrict__ lo,
                                                              int64_t ld_dst) {
  pdl_wait();
  pdl_trigger();
  __shared__ float tile[64][65];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int tiles_c = (cols + 63) / 64;
  const int64_t tiles = (int64_t)((rows + 63) / 64) * tiles_c;
  for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
    const int r0 = (int)(t / tiles_c) * 64, c0 = (int)(t % tiles_c) * 64;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const int rr = ty + 16 * p, r = r0 + rr;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = c0 + 4 * tx + e;
        tile[rr][4 * tx + e] = (r < rows && c < cols) ? src[(int64_t)r * ld_src + c] : 0.f;
      }
    }
    __syncthreads();
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const int cc = ty + 16 * p, c = c0 + cc, r = r0 + 4 * tx;
      if (c < cols) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (r + e >= rows) continue;
          float h, l;
          tf32_split(tile[4 * tx + e][cc], h, l);
          hi[(int64_t)c * ld_dst + r + e] = h;
          lo[(int64_t)c * ld_dst + r + e] = l;
        }
      }
    }
    __syncthreads();
  }
}

cudaError_t launch_split_tf32(bool transpose, int rows, int cols, const float* src,
                              int64_t ld_src, float* hi, float* lo, int64_t ld_dst,
                              LaunchCtx& ctx) {
  cudaError_t e;
  if (!transpose) {
    if ((ld_dst % 4) != 0 || ((reinterpret_cast<uintptr_t>(hi) | reinterpret_cast<uintptr_t>(lo)) & 15u))
      return cudaErrorInvalidValue;
    const int grid = grid_for((int64_t)rows * (ld_dst / 4), 256);
    e = launch_kernel(split_rows_kernel, dim3(grid), dim3(256), 0, ctx.stream, 1, rows, cols, src,
                      ld_src, hi, lo, ld_dst);
  } else {
    const int64_t tiles = (int64_t)((rows + 63) / 64) * ((cols + 63) / 64);
    const int grid = grid_for(tiles * 256, 256);
    e = launch_kernel(split_transpose_kernel, dim3(grid), dim3(256), 0, ctx.stream, 1, rows, cols,
                      src, ld_src, hi, lo, ld_dst);
  }
  if (e == cudaSuccess) ctx.launches++;
  return e;
}

cudaError_t launch_repack_32(int rows, int cols, const void* src, int64_t ld_src, void* dst,
                             int64_t ld_dst, LaunchCtx& ctx) {
  return launch_repack<uint32_t>(rows, cols, src, ld_src, dst, ld_dst, ctx);
}

cudaError_t launch_transpose_f32(int rows, int cols, const float* src, int64_t ld_src,
                                 float* dst, int64_t ld_dst, LaunchCtx& ctx) {
  const int64_t tiles = (int64_t)((rows + 63) / 64) * ((cols + 63) / 64);
  const int grid = grid_for(tiles * 256, 256);
  // 128-bit accesses need 16-byte aligned rows on both sides
  const bool vec = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15u) == 0 &&
                   (ld_src % 4) == 0 && (ld_dst % 4) == 0;
  cudaError_t e = vec ? launch_kernel(transpose_f32_kernel<true>, dim3(grid), dim3(256), 0,
                                      ctx.stream, 1, rows, cols, src, ld_src, dst, ld_dst)
                       : launch_kernel(transpose_f32_kernel<false>, dim3(grid), dim3(256), 0,
                                      ctx.stream, 1, rows, cols, src, ld_src, dst, ld_dst);
  if (e == cudaSuccess) ctx.launches++;
  return e;
}

cudaError_t launch_splitk_reduce(int dtype, int M, int N, int splits, const float* P, void* C,
                                 int64_t ldc, float alpha, float beta, LaunchCtx& ctx,
                                 Epilogue ep) {
  const int threads = 256;
  const bool vec = (N % 4) == 0;
  const int64_t items = vec ? (int64_t)M * (N / 4) : (int64_t)M * N;
  const int grid = grid_for(items, threads);
  const dim3 g(grid), b(threads);
  cudaError_t e;
  if (dtype == 0) {
    e = vec ? launch_kernel(splitk_reduce_vec4<float>, g, b, 0, ctx.stream, 1, M, N, splits, P,
                            (float*)C, ldc, alpha, beta, ep)
            : launch_kernel(splitk_reduce_scalar<float>, g, b, 0, ctx.stream, 1, M, N, splits, P,
                            (float*)C, ldc, alpha, beta, ep);
  } else if (dtype == 1) {
    e = vec ? launch_kernel(splitk_reduce_vec4<__half>, g, b, 0, ctx.stream, 1, M, N, splits, P,
                            (__half*)C, ldc, alpha, beta, ep)
            : launch_kernel(splitk_reduce_scalar<__half>, g, b, 0, ctx.stream, 1, M, N, splits, P,
                            (__half*)C, ldc, alpha, beta, ep);
  } else {
    e = vec ? launch_kernel(splitk_reduce_vec4<__nv_bfloat16>, g, b, 0, ctx.stream, 1, M, N, splits,
                            P, (__nv_bfloat16*)C, ldc, alpha, beta, ep)
            : launch_kernel(splitk_reduce_scalar<__nv_bfloat16>, g, b, 0, ctx.stream, 1, M, N,
                            splits, P, (__nv_bfloat16*)C, ldc, alpha, beta, ep);
  }
  if (e == cudaSuccess) ctx.launches++;
  return e;
}

cudaError_t launch_scale(int dtype, int M, int N, void* C, int64_t ldc, float beta,
                         LaunchCtx& ctx, Epilogue ep) {
  const int threads = 256;
  const int grid = grid_for((int64_t)M * N, threads);
  const dim3 g(grid), b(threads);
  cudaError_t e;
  if (dtype == 0)
    e = launch_kernel(scale_kernel<float>, g, b, 0, ctx.stream, 1, M, N, (float*)C, ldc, beta, ep);
  else if (dtype == 1)
    e = launch_kernel(scale_kernel<__half>, g, b, 0, ctx.stream, 1, M, N, (__half*)C, ldc, beta, ep);
  else
    e = launch_kernel(scale_kernel<__nv_bfloat16>, g, b, 0, ctx.stream, 1, M, N,
                      (__nv_bfloat16*)C, ldc, beta, ep);
  if (e == cudaSuccess) ctx.launches++;
  return e;
}

cudaError_t launch_repack_16(int rows, int cols, const void* src, int64_t ld_src, void* dst,
                             int64_t ld_dst, LaunchCtx& ctx) {
  return launch_repack<uint16_t>(rows, cols, src, ld_src, dst, ld_dst, ctx);
}

}  // namespace gb300
