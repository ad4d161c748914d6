// Host-side TMA descriptors (CUtensorMap) for the packed weights and scales.
//
// The driver function that encodes a descriptor is looked up once through the runtime, so the
// library does not link against libcuda (it still loads on machines without a GPU driver).
// Descriptors embed the global address, so they are built per call; a small per-thread cache
// returns the previous descriptor when the same tensor is used again.
#include <cuda.h>
#include <cuda_runtime.h>
#include <string.h>

#include <mutex>

#include "internal.h"

namespace w4a16 {
namespace {

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_status = cudaSuccess;

void load_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                   cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
    g_encode_status = (e != cudaSuccess) ? e : cudaErrorNotSupported;
    return;
  }
  g_encode = reinterpret_cast<EncodeFn>(fn);
}

struct CacheEntry {
  const void* ptr;
  uint64_t d0, d1, d2;
  uint32_t b0, b1;
  int dtype, swz;
  CUtensorMap map;
};
constexpr int kCacheSize = 8;
thread_local CacheEntry t_cache[kCacheSize];
thread_local int t_next = 0;

}  // namespace

// 3-D tiled descriptor of a row-major [d2][d1][d0] tensor (d0 contiguous), box (b0 x b1 x 1).
cudaError_t make_tmap_ex(CUtensorMap* out, CUtensorMapDataType dtype, uint32_t elem_bytes,
                         CUtensorMapSwizzle swz, const void* base, uint64_t d0, uint64_t d1,
                         uint64_t d2, uint32_t b0, uint32_t b1) {
  for (int i = 0; i < kCacheSize; ++i) {
    const CacheEntry& c = t_cache[i];
    if (c.ptr == base && c.d0 == d0 && c.d1 == d1 && c.d2 == d2 && c.b0 == b0 && c.b1 == b1 &&
        c.dtype == (int)dtype && c.swz == (int)swz) {
      *out = c.map;
      return cudaSuccess;
    }
  }
  std::call_once(g_encode_once, load_encode);
  if (!g_encode) return g_encode_status;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {d0 * elem_bytes, d0 * d1 * elem_bytes};
  const cuuint32_t box[3] = {b0, b1, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  CUtensorMap m;
  memset(&m, 0, sizeof(m));
  const CUresult r = g_encode(&m, dtype, 3, const_cast<void*>(base), dims, strides, box, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  CacheEntry& c = t_cache[t_next];
  t_next = (t_next + 1) % kCacheSize;
  c.ptr = base;
  c.d0 = d0;
  c.d1 = d1;
  c.d2 = d2;
  c.b0 = b0;
  c.b1 = b1;
  c.dtype = (int)dtype;
  c.swz = (int)swz;
  c.map = m;
  *out = m;
  return cudaSuccess;
}

// Tiled descriptor of `rank` (2..5) dimensions with explicit byte strides of dimensions 1..rank-1
// (any order: a dimension may step through memory faster than the one before it) and box
// `box[0..rank-1]`. Out-of-range box elements read as zero. Not cached: callers build these once
// per launch.
cudaError_t make_tmap_nd(CUtensorMap* out, CUtensorMapDataType dtype, CUtensorMapSwizzle swz,
                         const void* base, int rank, const uint64_t* dims,
                         const uint64_t* strides, const uint32_t* box) {
  if (rank < 2 || rank > 5) return cudaErrorInvalidValue;
  std::call_once(g_encode_once, load_encode);
  if (!g_encode) return g_encode_status;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    es[i] = 1;
    if (i > 0) st[i - 1] = strides[i - 1];
  }
  memset(out, 0, sizeof(*out));
  const CUresult r = g_encode(out, dtype, (cuuint32_t)rank, const_cast<void*>(base), d, st, b, es,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// kind 0: packed codes (int32, 128-byte swizzle); kind 1: scales (float32, no swizzle).
cudaError_t make_tmap(CUtensorMap* out, int kind, const void* base, uint64_t d0, uint64_t d1,
                      uint64_t d2, uint32_t b0, uint32_t b1) {
  return make_tmap_ex(out,
                      kind == 0 ? CU_TENSOR_MAP_DATA_TYPE_INT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                      4, kind == 0 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, base,
                      d0, d1, d2, b0, b1);
}

}  // namespace w4a16
