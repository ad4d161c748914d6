// Small-M (decode / draft-tree verify) weight-streaming GEMM: y = x @ dequant(W), float32
// activations and output (also in a bf16 form: bf16 activations and output, M <= 16).
//
// Page "The Weight of Precision: Building Native INT4 Quantization for a Custom Speculative
// Decoding Engine", section "The Kernel: w4a16_gemm" (FP32 activations, packed INT4 weights,
// group-32 float32 scales); the pages measure the optimized kernel against HBM bandwidth, so the
// design goal is to stream every packed weight and scale byte exactly once.
//
// Grid: x = tiles of kWN slices (one warp per slice of 32 or 64 weight columns), y = CK slices
// of K, z = 16-row slices of M (one for M <= 16). The CK CTAs of one tile form a thread-block
// cluster and add their partial tiles through distributed shared memory in rank order:
// deterministic, no global scratch, no atomics.
// The per-warp main loop lives in mma_core.cuh.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "internal.h"
#include "mma_core.cuh"
#include "splitk.cuh"

namespace cg = cooperative_groups;

namespace w4a16 {
namespace {

using namespace mma;

// Geometry of the two orientations.
//   up to 8 rows : A = codes; 4-warp CTAs, 2-stage rings and a 12-16 KB activation budget keep
//                  a CTA near 53 KB so four fit per SM (16 warps, ~80 KB of copies in flight);
//   9..16 rows   : A = activations (no padded MMA rows); 4-warp CTAs, 3-stage rings, 16 KB.
constexpr int kWN = 4;  // warps (slices) per CTA

// Tuning knobs (compile-time; defaults are the measured best on GB300).
#ifndef W4A16_CODES_RING
#define W4A16_CODES_RING 2
#endif
#ifndef W4A16_CODES_MINB
#define W4A16_CODES_MINB 4
#endif
#ifndef W4A16_ACTS_RING
#define W4A16_ACTS_RING 3
#endif
#ifndef W4A16_ACTS_MINB
#define W4A16_ACTS_MINB 4
#endif
#ifndef W4A16_WIDE_CH
#define W4A16_WIDE_CH 4
#endif
#ifndef W4A16_B16_WIDE_CH
#define W4A16_B16_WIDE_CH 4
#endif

template <int NB, int CH>
using CodesGeo = Geo<NB, CH, kWN, W4A16_CODES_RING, NB == 1 ? 12288 : 16384>;
template <int CH>
using ActsGeo = Geo<4, CH, kWN, W4A16_ACTS_RING, 16384>;

// Grid z = 16-row slices of a larger M (x and y advance by 16 rows per slice): the first row of
// this CTA's slice and the slice's row count.
__device__ __forceinline__ size_t slice_row0() { return (size_t)blockIdx.z * kGemvMaxM; }
__device__ __forceinline__ int slice_rows(int M) {
  return min(M - (int)blockIdx.z * kGemvMaxM, kGemvMaxM);
}

template <int NB, int CH, bool SWIGLU>
__global__ void __launch_bounds__(kWN * 32, W4A16_CODES_MINB)
    gemv_codes_kernel(const __grid_constant__ CUtensorMap tq,
                      const __grid_constant__ CUtensorMap ts, const float* __restrict__ x,
                      float* __restrict__ y, int M, int N, int K, unsigned int* err) {
  using L = CodesGeo<NB, CH>;
  extern __shared__ __align__(1024) char smem_raw[];
  char* smem = align1024(smem_raw);
  x += slice_row0() * K;
  y += slice_row0() * (SWIGLU ? N / 2 : N);
  M = slice_rows(M);
  cg::cluster_group cluster = cg::this_cluster();
  const int tile = blockIdx.x;
  const int CK = (int)cluster.dim_blocks().y;
  const int rank = (int)cluster.block_index().y;
  const int warp = threadIdx.x >> 5;
  const int G = K / kGroup;
  const int q0 = (int)((long long)rank * G / CK);
  const int q1 = (int)((long long)(rank + 1) * G / CK);

  init_barriers<L>(smem, kWN);
  float acc[CH][2][NB][4];
  int seq = 0;
  auto rowptr = [&](int m) { return x + (size_t)m * K; };
  stream_groups<NB, CH, SWIGLU, kWN, L>(rowptr, M, &tq, &ts, 0, N, q0, q1 - q0, tile * kWN,
                                        smem, seq, err, acc);
  if (CK == 1) {
    store_direct<NB, CH, SWIGLU>(acc, tile * kWN + warp, N, M, y);
    return;
  }
  constexpr int kCols = kWN * 32 * CH;
  static_assert(4 * NB * kCols * 4 <= kWN * L::kRing * CH * L::kCodeTile,
                "split-K tile must fit in the code ring");
  float* red = reinterpret_cast<float*>(smem + L::kCodeOff);
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int c = 0; c < CH; ++c)
#pragma unroll
    for (int b = 0; b < NB; ++b)
      *reinterpret_cast<float4*>(&red[(4 * b + t) * kCols +
                                      tile_local_col<CH, SWIGLU, kWN>(warp, c, g)]) =
          chunk_result<NB, CH>(acc, c, b);
  cluster_finish<SWIGLU, kCols>(cluster, red, tile, M, N, y);
}

template <int CH, bool SWIGLU>
__global__ void __launch_bounds__(kWN * 32, W4A16_ACTS_MINB)
    gemv_acts_kernel(const __grid_constant__ CUtensorMap tq,
                     const __grid_constant__ CUtensorMap ts, const float* __restrict__ x,
                     float* __restrict__ y, int M, int N, int K, unsigned int* err) {
  using L = ActsGeo<CH>;
  extern __shared__ __align__(1024) char smem_raw[];
  char* smem = align1024(smem_raw);
  x += slice_row0() * K;
  y += slice_row0() * (SWIGLU ? N / 2 : N);
  M = slice_rows(M);
  cg::cluster_group cluster = cg::this_cluster();
  const int tile = blockIdx.x;
  const int CK = (int)cluster.dim_blocks().y;
  const int rank = (int)cluster.block_index().y;
  const int warp = threadIdx.x >> 5;
  const int G = K / kGroup;
  const int q0 = (int)((long long)rank * G / CK);
  const int q1 = (int)((long long)(rank + 1) * G / CK);

  init_barriers<L>(smem, kWN);
  float acc[CH][4][4];
  int seq = 0;
  auto rowptr = [&](int m) { return x + (size_t)m * K; };
  stream_groups_xa<CH, SWIGLU, kWN, L>(rowptr, M, &tq, &ts, 0, N, q0, q1 - q0, tile * kWN, smem,
                                       seq, err, acc);
  if (CK == 1) {
    store_direct_xa<CH, SWIGLU>(acc, tile * kWN + warp, N, M, y);
    return;
  }
  constexpr int kCols = kWN * 32 * CH;
  static_assert(16 * kCols * 4 <= kWN * L::kRing * CH * L::kCodeTile,
                "split-K tile must fit in the code ring");
  float* red = reinterpret_cast<float*>(smem + L::kCodeOff);
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int hh[2] = {lane_chunk(2 * t), lane_chunk(2 * t + 1)};
#pragma unroll
  for (int c = 0; c < CH; ++c)
#pragma unroll
    for (int hf = 0; hf < 2; ++hf)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        // tile_local_col with the lane chunk of B column 2t + e
        int lc;
        if (SWIGLU) {
          constexpr int H = CH / 2;
          lc = (c >= H ? kWN * 16 * CH : 0) + warp * 16 * CH + 32 * (c >= H ? c - H : c) +
               4 * hh[e];
        } else {
          lc = warp * 32 * CH + 32 * c + 4 * hh[e];
        }
        *reinterpret_cast<float4*>(&red[(g + 8 * hf) * kCols + lc]) = xa_result<CH>(acc, c, hf, e);
      }
  cluster_finish<SWIGLU, kCols>(cluster, red, tile, M, N, y);
}

// bf16 activations (x[M, K] bf16, y[M, N] bf16, M <= 16): the codes orientation with x rows as
// MMA columns, 8 rows per n8 block. Lane (g, t) ends with rows 8b + 2t and 8b + 2t + 1 of n8 block
// b; for each of them the lane's 4 columns 4 h(g) + 0..3 of tile c are below.
template <int NB, int CH>
__device__ __forceinline__ float4 b16_result(const float (&acc)[CH][2][NB][4], int c, int b,
                                             int odd) {
  return make_float4(acc[c][0][b][odd], acc[c][0][b][2 + odd], acc[c][1][b][odd],
                     acc[c][1][b][2 + odd]);
}

template <int NB, int CH>
__global__ void __launch_bounds__(kWN * 32, W4A16_CODES_MINB)
    gemv_b16_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap ts,
                    const uint16_t* __restrict__ x, uint16_t* __restrict__ y, int M, int N, int K,
                    unsigned int* err) {
  using L = CodesGeo<NB, CH>;
  extern __shared__ __align__(1024) char smem_raw[];
  char* smem = align1024(smem_raw);
  x += slice_row0() * K;  // M <= 16: one slice
  y += slice_row0() * N;
  M = slice_rows(M);
  cg::cluster_group cluster = cg::this_cluster();
  const int tile = blockIdx.x;
  const int CK = (int)cluster.dim_blocks().y;
  const int rank = (int)cluster.block_index().y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int G = K / kGroup;
  const int q0 = (int)((long long)rank * G / CK);
  const int q1 = (int)((long long)(rank + 1) * G / CK);

  init_barriers<L>(smem, kWN);
  float acc[CH][2][NB][4];
  int seq = 0;
  auto rowptr = [&](int m) { return x + (size_t)m * K; };
  stream_groups<NB, CH, false, kWN, L, true>(rowptr, M, &tq, &ts, 0, N, q0, q1 - q0, tile * kWN,
                                             smem, seq, err, acc);
  if (CK == 1) {
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      bool valid;
      const int col = out_col<CH, false>(tile * kWN + warp, c, g, N, &valid);
      if (!valid) continue;
#pragma unroll
      for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int odd = 0; odd < 2; ++odd) {
          const int m = 8 * b + 2 * t + odd;
          if (m < M) {
            const float4 v = b16_result<NB, CH>(acc, c, b, odd);
            const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
            const __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
            uint2 o;
            o.x = *reinterpret_cast<const uint32_t*>(&lo);
            o.y = *reinterpret_cast<const uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(y + (size_t)m * N + col) = o;
          }
        }
    }
    return;
  }
  constexpr int kCols = kWN * 32 * CH;
  static_assert(8 * NB * kCols * 4 <= kWN * L::kRing * CH * L::kCodeTile,
                "split-K tile must fit in the code ring");
  float* red = reinterpret_cast<float*>(smem + L::kCodeOff);
#pragma unroll
  for (int c = 0; c < CH; ++c)
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
      for (int odd = 0; odd < 2; ++odd)
        *reinterpret_cast<float4*>(&red[(8 * b + 2 * t + odd) * kCols +
                                        tile_local_col<CH, false, kWN>(warp, c, g)]) =
            b16_result<NB, CH>(acc, c, b, odd);
  cluster_finish<false, kCols, uint16_t>(cluster, red, tile, M, N, y);
}

constexpr int kMaxCluster = 16;

struct LaunchData {
  int occ;
  int max_clusters[kMaxCluster + 1];  // index = cluster size
};
using LaunchCache = PerDeviceOnce<LaunchData>;

// Slices (one warp each) of a problem for CH tiles per warp.
template <int CH, bool SWIGLU>
int slices_of(int N) {
  return SWIGLU ? ((N >> 1) + 16 * CH - 1) / (16 * CH) : (N + 32 * CH - 1) / (32 * CH);
}

// A kernel's resident CTAs per SM and, per cluster size, its resident clusters (queried once per
// device).
template <typename Kern>
cudaError_t launch_data(Kern kern, int smem, LaunchCache& cache, const DeviceInfo& di,
                        const LaunchData** out) {
  return cache.get(di.device, [&](LaunchData& d) {
    cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (r != cudaSuccess) return r;
    r = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (r != cudaSuccess) return r;
    int occ = 0;
    r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kWN * 32, smem);
    if (r != cudaSuccess) return r;
    d.occ = occ < 1 ? 1 : occ;
    for (int ck = 1; ck <= kMaxCluster; ck *= 2) {
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
      d.max_clusters[ck] = nc;
    }
    return cudaSuccess;
  }, out);
}

// Split-K factor for `units` clusters' worth of tiles (x row slices): the CK whose waves of
// resident clusters fill the GPU's CTA slots most evenly, each CTA keeping at least 8 groups of K.
// *eff = the filled fraction of the slots over those waves.
inline int plan_split(const LaunchData& ld, long long units, int G, const DeviceInfo& di,
                      double* eff) {
  const double slots = (double)di.sm_count * ld.occ;
  int CK = 1;
  double best = -1.0;
  for (int ck = 1; ck <= kMaxCluster; ck *= 2) {
    if (ck > 1 && G / ck < 8) break;
    const int nc = ld.max_clusters[ck];
    if (nc <= 0) continue;
    const long long waves = (units + nc - 1) / nc;
    const double e = (double)units * ck / ((double)waves * slots);
    if (e > best * 1.03) {
      best = e;
      CK = ck;
    }
  }
  if (eff) *eff = best;
  return CK;
}

// Launches `kern` over tiles x CK clusters x 16-row slices of M.
template <typename Kern, typename XT, typename YT>
cudaError_t launch_split(Kern kern, int smem, LaunchCache& cache, int tiles, const XT* x,
                         const int32_t* qw, const float* sc, YT* y, int M, int N, int K,
                         const DeviceInfo& di, cudaStream_t s) {
  const int nz = (M + kGemvMaxM - 1) / kGemvMaxM;  // 16-row slices, grid z
  const LaunchData* ld = nullptr;
  cudaError_t e = launch_data(kern, smem, cache, di, &ld);
  if (e != cudaSuccess) return e;
  const int CK = plan_split(*ld, (long long)tiles * nz, K / kGroup, di, nullptr);
  CUtensorMap tq, ts;
  e = make_tmap(&tq, 0, qw, (uint64_t)N, (uint64_t)(K / 8), 1, 32, kRows);
  if (e != cudaSuccess) return e;
  e = make_tmap(&ts, 1, sc, (uint64_t)N, (uint64_t)(K / kGroup), 1, 32, kRows / 4);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles, CK, nz);
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
  return cudaLaunchKernelEx(&cfg, kern, tq, ts, x, y, M, N, K, device_error_word());
}

// One launch cache per kernel instantiation.
template <int NB, int CH, bool SWIGLU>
LaunchCache codes_cache;
template <int CH, bool SWIGLU>
LaunchCache acts_cache;
template <int NB, int CH>
LaunchCache b16_cache;

template <int NB, int CH, bool SWIGLU>
cudaError_t launch_codes(const float* x, const int32_t* qw, const float* sc, float* y, int M,
                         int N, int K, const DeviceInfo& di, cudaStream_t s) {
  const int tiles = (slices_of<CH, SWIGLU>(N) + kWN - 1) / kWN;
  return launch_split(gemv_codes_kernel<NB, CH, SWIGLU>, CodesGeo<NB, CH>::kAlloc,
                      codes_cache<NB, CH, SWIGLU>, tiles, x, qw, sc, y, M, N, K, di, s);
}

template <int CH, bool SWIGLU>
cudaError_t launch_acts(const float* x, const int32_t* qw, const float* sc, float* y, int M,
                        int N, int K, const DeviceInfo& di, cudaStream_t s) {
  const int tiles = (slices_of<CH, SWIGLU>(N) + kWN - 1) / kWN;
  return launch_split(gemv_acts_kernel<CH, SWIGLU>, ActsGeo<CH>::kAlloc, acts_cache<CH, SWIGLU>,
                      tiles, x, qw, sc, y, M, N, K, di, s);
}

// Whether 4 tiles per warp (128 columns) fill the GPU at least about as well as 2: each width's
// tiles with the split-K factor its resident clusters allow (plan_split). Wide tiles halve the
// CTAs but share each activation fragment between more columns, so they win ties.
template <typename KernW, typename KernN>
cudaError_t prefer_wide(KernW kw, int smem_w, LaunchCache& cw, int tiles_w, KernN kn, int smem_n,
                        LaunchCache& cn, int tiles_n, int K, const DeviceInfo& di, bool* wide) {
  const LaunchData *lw = nullptr, *ln = nullptr;
  cudaError_t e = launch_data(kw, smem_w, cw, di, &lw);
  if (e != cudaSuccess) return e;
  e = launch_data(kn, smem_n, cn, di, &ln);
  if (e != cudaSuccess) return e;
  double ew = 0.0, en = 0.0;
  (void)plan_split(*lw, tiles_w, K / kGroup, di, &ew);
  (void)plan_split(*ln, tiles_n, K / kGroup, di, &en);
  *wide = ew * 1.03 >= en;
  return cudaSuccess;
}

// Up to 4 rows: 4 or 2 tiles per warp (prefer_wide); 5..8 rows: 2; 9 rows and more: the
// activations-as-A kernel, 2 tiles, one 16-row slice per grid z (all slices in one launch, so CTAs
// of several slices stream the same weight tiles at about the same time and share them through
// L2).
template <bool SWIGLU>
cudaError_t dispatch(const float* x, const int32_t* qw, const float* sc, float* y, int M, int N,
                     int K, const DeviceInfo& di, cudaStream_t s) {
  if (M <= 4) {
    constexpr int W = W4A16_WIDE_CH;
    bool wide = true;
    const cudaError_t e = prefer_wide(
        gemv_codes_kernel<1, W, SWIGLU>, CodesGeo<1, W>::kAlloc, codes_cache<1, W, SWIGLU>,
        (slices_of<W, SWIGLU>(N) + kWN - 1) / kWN, gemv_codes_kernel<1, 2, SWIGLU>,
        CodesGeo<1, 2>::kAlloc, codes_cache<1, 2, SWIGLU>,
        (slices_of<2, SWIGLU>(N) + kWN - 1) / kWN, K, di, &wide);
    if (e != cudaSuccess) return e;
    return wide ? launch_codes<1, W, SWIGLU>(x, qw, sc, y, M, N, K, di, s)
                : launch_codes<1, 2, SWIGLU>(x, qw, sc, y, M, N, K, di, s);
  }
  if (M <= 8) return launch_codes<2, 2, SWIGLU>(x, qw, sc, y, M, N, K, di, s);
  return launch_acts<2, SWIGLU>(x, qw, sc, y, M, N, K, di, s);  // 9+ rows, 16 per grid z
}

template <int NB, int CH>
cudaError_t launch_b16(const uint16_t* x, const int32_t* qw, const float* sc, uint16_t* y, int M,
                       int N, int K, const DeviceInfo& di, cudaStream_t s) {
  const int tiles = (slices_of<CH, false>(N) + kWN - 1) / kWN;
  return launch_split(gemv_b16_kernel<NB, CH>, CodesGeo<NB, CH>::kAlloc, b16_cache<NB, CH>, tiles,
                      x, qw, sc, y, M, N, K, di, s);
}

}  // namespace

cudaError_t launch_gemv_b16(const uint16_t* x, const int32_t* qw, const float* sc, uint16_t* y,
                            int M, int N, int K, cudaStream_t s) {
  DeviceInfo di;
  cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return e;
  if (M <= 8) {
    constexpr int W = W4A16_B16_WIDE_CH;
    bool wide = true;
    e = prefer_wide(gemv_b16_kernel<1, W>, CodesGeo<1, W>::kAlloc, b16_cache<1, W>,
                    (slices_of<W, false>(N) + kWN - 1) / kWN, gemv_b16_kernel<1, 2>,
                    CodesGeo<1, 2>::kAlloc, b16_cache<1, 2>,
                    (slices_of<2, false>(N) + kWN - 1) / kWN, K, di, &wide);
    if (e != cudaSuccess) return e;
    return wide ? launch_b16<1, W>(x, qw, sc, y, M, N, K, di, s)
                : launch_b16<1, 2>(x, qw, sc, y, M, N, K, di, s);
  }
  if (M <= 16) return launch_b16<2, 2>(x, qw, sc, y, M, N, K, di, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_gemv(const float* x, const int32_t* qw, const float* sc, float* y, int M,
                        int N, int K, bool swiglu, cudaStream_t s) {
  DeviceInfo di;
  cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return e;
  return swiglu ? dispatch<true>(x, qw, sc, y, M, N, K, di, s)
                : dispatch<false>(x, qw, sc, y, M, N, K, di, s);
}

}  // namespace w4a16
