// Small-M (decode / draft-tree verify) weight-streaming GEMM: y = x @ dequant(W), float32.
//
// Page "The Weight of Precision: Building Native INT4 Quantization for a Custom Speculative
// Decoding Engine", section "The Kernel: w4a16_gemm" (FP32 activations, packed INT4 weights,
// group-32 float32 scales); the pages measure the optimized kernel against HBM bandwidth, so the
// design goal is to stream every packed weight and scale byte exactly once.
//
// Grid: x = 128-column tiles, y = S slices of K. The S CTAs of one tile form a thread-block
// cluster and add their partial tiles through distributed shared memory in rank order, so the
// result is deterministic and needs no global scratch or atomics.
#include <cooperative_groups.h>

#include "internal.h"
#include "simt_core.cuh"

namespace cg = cooperative_groups;

namespace w4a16 {
namespace {

using namespace simt;

template <int M, bool SWIGLU>
__global__ void __launch_bounds__(kThreads) gemv_simt_kernel(const float* __restrict__ x,
                                                             const int32_t* __restrict__ qw,
                                                             const float* __restrict__ sc,
                                                             float* __restrict__ y, int N, int K) {
  extern __shared__ float4 smem4[];
  float* red = reinterpret_cast<float*>(smem4);  // [kWarps][M][kTileN]
  cg::cluster_group cluster = cg::this_cluster();
  const int tile = blockIdx.x;
  const int S = (int)cluster.dim_blocks().y;
  const int rank = (int)cluster.block_index().y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  int col;
  bool valid;
  lane_columns<SWIGLU>(tile, lane, N, &col, &valid);
  const int G = K / kGroup;
  const int g0 = (int)((long long)rank * G / S);
  const int g1 = (int)((long long)(rank + 1) * G / S);

  float acc[M][4];
#pragma unroll
  for (int m = 0; m < M; ++m)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[m][c] = 0.0f;
  if (valid) {
    const float* xrow[M];
#pragma unroll
    for (int m = 0; m < M; ++m) xrow[m] = x + (size_t)m * K;
    accumulate_groups<M>(xrow, qw, sc, N, col, g0 + warp, g1, kWarps, acc);
  }
  reduce_warps<M>(red, acc, warp, lane);

  // Cross-CTA (split-K) reduction over the cluster, in rank order.
  if (S > 1) cluster.sync();
  if (SWIGLU) {
    const int I = N >> 1;
    const int per = 64 / S;
    for (int idx = threadIdx.x; idx < M * per; idx += kThreads) {
      const int m = idx / per;
      const int j = rank * per + (idx - m * per);
      float gsum = 0.0f, usum = 0.0f;
      for (int q = 0; q < S; ++q) {
        const float* r = (S > 1) ? cluster.map_shared_rank(red, q) : red;
        gsum += r[m * kTileN + j];
        usum += r[m * kTileN + 64 + j];
      }
      const int o = 64 * tile + j;
      if (o < I) y[(size_t)m * I + o] = silu_f(gsum) * usum;
    }
  } else {
    const int per = kTileN / S;
    for (int idx = threadIdx.x; idx < M * per; idx += kThreads) {
      const int m = idx / per;
      const int j = rank * per + (idx - m * per);
      float sum = 0.0f;
      for (int q = 0; q < S; ++q) {
        const float* r = (S > 1) ? cluster.map_shared_rank(red, q) : red;
        sum += r[m * kTileN + j];
      }
      const int o = kTileN * tile + j;
      if (o < N) y[(size_t)m * N + o] = sum;
    }
  }
  if (S > 1) cluster.sync();  // peers may still read this CTA's shared memory
}

struct KernelCache {
  int occ = 0;
  int attr_devices = 0;  // bitmask of devices with the shared-memory attribute set
};

template <int M, bool SWIGLU>
cudaError_t launch_m(const float* x, const int32_t* qw, const float* sc, float* y, int N, int K,
                     const DeviceInfo& di, cudaStream_t s) {
  static KernelCache cache;
  auto kern = gemv_simt_kernel<M, SWIGLU>;
  const size_t smem = (size_t)kWarps * M * kTileN * sizeof(float);
  const int bit = 1 << (di.device & 31);
  if (!(cache.attr_devices & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, smem);
    if (e != cudaSuccess) return e;
    cache.occ = occ < 1 ? 1 : occ;
    cache.attr_devices |= bit;
  }
  const int tiles = SWIGLU ? ((N >> 1) + 63) / 64 : (N + kTileN - 1) / kTileN;
  const int G = K / kGroup;
  // Split K over a cluster of S CTAs when the tiles alone cannot fill the GPU evenly.
  const long long slots = (long long)di.sm_count * cache.occ;
  int S = 1;
  double best = 0.0;
  for (int cand = 1; cand <= 8; cand *= 2) {
    if (cand > 1 && G / cand < 2) break;
    const long long ctas = (long long)tiles * cand;
    const long long waves = (ctas + slots - 1) / slots;
    const double eff = (double)ctas / (double)(waves * slots);
    if (eff > best + 0.03) {
      best = eff;
      S = cand;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles, S, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = S;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, x, qw, sc, y, N, K);
}

template <bool SWIGLU>
cudaError_t dispatch_m(const float* x, const int32_t* qw, const float* sc, float* y, int M, int N,
                       int K, const DeviceInfo& di, cudaStream_t s) {
  switch (M) {
#define W4A16_CASE(mm) \
  case mm:             \
    return launch_m<mm, SWIGLU>(x, qw, sc, y, N, K, di, s);
    W4A16_CASE(1) W4A16_CASE(2) W4A16_CASE(3) W4A16_CASE(4) W4A16_CASE(5) W4A16_CASE(6)
    W4A16_CASE(7) W4A16_CASE(8) W4A16_CASE(9) W4A16_CASE(10) W4A16_CASE(11) W4A16_CASE(12)
    W4A16_CASE(13) W4A16_CASE(14) W4A16_CASE(15) W4A16_CASE(16)
#undef W4A16_CASE
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_gemv(const float* x, const int32_t* qw, const float* sc, float* y, int M,
                        int N, int K, bool swiglu, cudaStream_t s) {
  DeviceInfo di;
  cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return e;
  return swiglu ? dispatch_m<true>(x, qw, sc, y, M, N, K, di, s)
                : dispatch_m<false>(x, qw, sc, y, M, N, K, di, s);
}

}  // namespace w4a16
