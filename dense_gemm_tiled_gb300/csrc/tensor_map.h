// Host side of the TMA tensor maps the GEMM kernels load through: the driver's
// encoding entry point and a per-thread cache of encoded maps.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gb300 {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    return (PFN_cuTensorMapEncodeTiled_v12000) nullptr;
  }();
  return fn;
}

// 3-D tensor map over `batch` row-major [rows, cols] matrices of `esize`-byte
// elements with row pitch `ld` and batch pitch `stride` elements; box = box_cols (inner) x
// box_rows x 1, 128-byte swizzle by default, out-of-range elements read as
// zero.  Returns false when the driver rejects the description (the launch
// then reports cudaErrorNotSupported and nothing runs).
//
// Encoded maps are kept in a small per-thread cache keyed by everything the
// description holds (address, element type and size, extents, pitches, box,
// swizzle): a map only describes a layout, so it stays valid for whatever
// memory lies at that address; a repeated call skips the encoding.
struct MapKey {
  const void* base;
  int64_t rows, cols, ld, batch, stride;
  int box_cols, box_rows, type, swizzle, esize;
  bool operator==(const MapKey& o) const {
    return base == o.base && rows == o.rows && cols == o.cols && ld == o.ld &&
           batch == o.batch && stride == o.stride && box_cols == o.box_cols &&
           box_rows == o.box_rows && type == o.type && swizzle == o.swizzle && esize == o.esize;
  }
};
struct MapEntry {
  MapKey key;
  CUtensorMap map;
  bool used;
};
constexpr int MAP_CACHE = 64;

inline uint64_t map_hash(const MapKey& k) {
  uint64_t h = (uint64_t)(uintptr_t)k.base * 0x9E3779B97F4A7C15ull;
  const int64_t v[9] = {k.rows, k.cols, k.ld, k.batch, k.stride, k.box_cols, k.box_rows,
                        k.type * 16 + k.swizzle, k.esize};
  for (int i = 0; i < 9; ++i) h = (h ^ (uint64_t)v[i]) * 0x100000001B3ull;
  return h ^ (h >> 29);
}

bool make_map(CUtensorMap* map, CUtensorMapDataType type, const void* base, int64_t rows,
              int64_t cols, int64_t ld, int box_cols, int box_rows,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B, int64_t batch = 1,
              int64_t stride = 0, int esize = 2) {
  // [batch][rows][cols]; a single matrix is batch 1 with a nominal pitch
  if (batch <= 1) stride = ld * (rows > 0 ? rows : 1);
  const MapKey key{base, rows, cols, ld, batch > 1 ? batch : 1, stride, box_cols, box_rows,
                   (int)type, (int)swizzle, esize};
  thread_local MapEntry cache[MAP_CACHE];
  MapEntry& slot = cache[map_hash(key) % MAP_CACHE];
  if (slot.used && slot.key == key) {
    *map = slot.map;
    return true;
  }
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)(batch > 1 ? batch : 1)};
  cuuint64_t strides[2] = {(cuuint64_t)(ld * esize), (cuuint64_t)(stride * esize)};
  cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, type, 3, const_cast<void*>(base), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  slot.key = key;
  slot.map = *map;
  slot.used = true;
  return true;
}

}  // namespace
}  // namespace gb300
