// Small-M (decode / draft-tree verify) weight-streaming GEMM: y = x @ dequant(W), float32.
//
// Page "The Weight of Precision: Building Native INT4 Quantization for a Custom Speculative
// Decoding Engine", section "The Kernel: w4a16_gemm" (FP32 activations, packed INT4 weights,
// group-32 float32 scales); the pages measure the optimized kernel against HBM bandwidth, so the
// design goal is to stream every packed weight and scale byte exactly once.
//
// Grid: x = tiles of kWN slices (32 weight columns each, one warp per slice), y = CK slices of
// K. The CK CTAs of one tile form a thread-block cluster and add their partial tiles through
// distributed shared memory in rank order: deterministic, no global scratch, no atomics.
// The per-warp main loop lives in mma_core.cuh.
#include <cooperative_groups.h>

#include "internal.h"
#include "mma_core.cuh"

namespace cg = cooperative_groups;

namespace w4a16 {
namespace {

using namespace mma;

constexpr int kWN = 8;  // warps (slices) per CTA

template <int NB, bool SWIGLU>
__global__ void __launch_bounds__(kWN * 32) gemv_mma_kernel(const float* __restrict__ x,
                                                            const int32_t* __restrict__ qw,
                                                            const float* __restrict__ sc,
                                                            float* __restrict__ y, int M, int N,
                                                            int K) {
  extern __shared__ __align__(128) char smem[];
  cg::cluster_group cluster = cg::this_cluster();
  const int tile = blockIdx.x;
  const int CK = (int)cluster.dim_blocks().y;
  const int rank = (int)cluster.block_index().y;
  const int warp = threadIdx.x >> 5;
  const int G = K / kGroup;
  const int q0 = (int)((long long)rank * G / CK);
  const int q1 = (int)((long long)(rank + 1) * G / CK);

  float acc[2][NB][4];
  auto rowptr = [&](int m) { return x + (size_t)m * K; };
  stream_groups<NB, SWIGLU, kWN>(rowptr, M, qw, sc, N, q0, q1 - q0, tile * kWN, smem, acc);

  if (CK == 1) {
    store_direct<NB, SWIGLU>(acc, tile * kWN + warp, N, M, y);
    return;
  }
  // Split-K: partial tile [4*NB rows][kWN*32 local columns] in shared memory (reusing the
  // cp.async rings), then rank r finishes its share of the columns over all ranks in order.
  constexpr int kCols = kWN * 32;
  float* red = reinterpret_cast<float*>(smem + Smem<NB, kWN>::kPipeOff);
  {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int h = (g >> 1) + 4 * (g & 1);
#pragma unroll
    for (int b = 0; b < NB; ++b)
      *reinterpret_cast<float4*>(&red[(4 * b + t) * kCols + warp * 32 + 4 * h]) =
          chunk_result<NB>(acc, b);
  }
  cluster.sync();
  if (SWIGLU) {
    // local output o (0 .. kWN*16-1): slice o/16, gate at local column 32 (o/16) + o%16,
    // up at 32 (o/16) + 16 + o%16 (chunks 0..3 are gate, 4..7 up).
    constexpr int kOut = kWN * 16;
    const int I = N >> 1;
    const int per = kOut / CK;
    for (int idx = threadIdx.x; idx < M * per; idx += blockDim.x) {
      const int m = idx / per;
      const int o = rank * per + (idx - m * per);
      const int lc = 32 * (o >> 4) + (o & 15);
      float gs = 0.0f, us = 0.0f;
      for (int q = 0; q < CK; ++q) {
        const float* r = cluster.map_shared_rank(red, q);
        gs += r[m * kCols + lc];
        us += r[m * kCols + lc + 16];
      }
      const int out = tile * kOut + o;
      if (out < I) y[(size_t)m * I + out] = silu_f(gs) * us;
    }
  } else {
    const int per = kCols / CK;
    for (int idx = threadIdx.x; idx < M * per; idx += blockDim.x) {
      const int m = idx / per;
      const int lc = rank * per + (idx - m * per);
      float s = 0.0f;
      for (int q = 0; q < CK; ++q) s += cluster.map_shared_rank(red, q)[m * kCols + lc];
      const int out = tile * kCols + lc;
      if (out < N) y[(size_t)m * N + out] = s;
    }
  }
  cluster.sync();  // peers may still be reading this CTA's shared memory
}

struct LaunchCache {
  int device_mask = 0;
  int occ = 0;
  int max_clusters[9] = {0};  // index = cluster size (1, 2, 4, 8)
};

template <int NB, bool SWIGLU>
cudaError_t launch_nb(const float* x, const int32_t* qw, const float* sc, float* y, int M, int N,
                      int K, const DeviceInfo& di, cudaStream_t s) {
  static LaunchCache cache;
  auto kern = gemv_mma_kernel<NB, SWIGLU>;
  constexpr int smem = Smem<NB, kWN>::kBytes;
  static_assert(4 * NB * kWN * 32 * 4 <= Smem<NB, kWN>::kPipeBytes, "split-K tile must fit");
  const int slices = SWIGLU ? ((N >> 1) + 15) / 16 : (N + 31) / 32;
  const int tiles = (slices + kWN - 1) / kWN;
  const int G = K / kGroup;
  const int bit = 1 << (di.device & 31);
  if (!(cache.device_mask & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kWN * 32, smem);
    if (e != cudaSuccess) return e;
    cache.occ = occ < 1 ? 1 : occ;
    for (int ck = 1; ck <= 8; ck *= 2) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(1, ck, 1);
      cfg.blockDim = dim3(kWN * 32, 1, 1);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = 1;
      at[0].val.clusterDim.y = ck;
      at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      int nc = 0;
      if (cudaOccupancyMaxActiveClusters(&nc, kern, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        nc = 0;
      }
      cache.max_clusters[ck] = nc;
    }
    cache.device_mask |= bit;
  }
  // Pick the K split whose waves of clusters fill the GPU most evenly.
  const double slots = (double)di.sm_count * cache.occ;
  int CK = 1;
  double best = -1.0;
  for (int ck = 1; ck <= 8; ck *= 2) {
    if (ck > 1 && G / ck < 4) break;
    const int nc = cache.max_clusters[ck];
    if (nc <= 0) continue;
    const long long waves = (tiles + nc - 1) / nc;
    const double eff = (double)tiles * ck / ((double)waves * slots);
    if (eff > best * 1.03) {
      best = eff;
      CK = ck;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles, CK, 1);
  cfg.blockDim = dim3(kWN * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = CK;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, x, qw, sc, y, M, N, K);
}

template <bool SWIGLU>
cudaError_t dispatch(const float* x, const int32_t* qw, const float* sc, float* y, int M, int N,
                     int K, const DeviceInfo& di, cudaStream_t s) {
  switch ((M + 3) / 4) {
    case 1: return launch_nb<1, SWIGLU>(x, qw, sc, y, M, N, K, di, s);
    case 2: return launch_nb<2, SWIGLU>(x, qw, sc, y, M, N, K, di, s);
    case 3: return launch_nb<3, SWIGLU>(x, qw, sc, y, M, N, K, di, s);
    case 4: return launch_nb<4, SWIGLU>(x, qw, sc, y, M, N, K, di, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_gemv(const float* x, const int32_t* qw, const float* sc, float* y, int M,
                        int N, int K, bool swiglu, cudaStream_t s) {
  DeviceInfo di;
  cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return e;
  return swiglu ? dispatch<true>(x, qw, sc, y, M, N, K, di, s)
                : dispatch<false>(x, qw, sc, y, M, N, K, di, s);
}

}  // namespace w4a16
