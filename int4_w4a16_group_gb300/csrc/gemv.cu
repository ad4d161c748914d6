// Small-M (decode / draft-tree verify) weight-streaming GEMM: y = x @ dequant(W), float32
// activations and output, optionally with the fused gate/up SwiGLU epilogue; and the bf16 form
// (bf16 activations and output, M <= 16).
//
// Page "The Weight of Precision: Building Native INT4 Quantization for a Custom Speculative
// Decoding Engine", section "The Kernel: w4a16_gemm" (FP32 activations, packed INT4 weights,
// group-32 float32 scales); the pages measure the optimized kernel against HBM bandwidth, so the
// design goal is to stream every packed weight and scale byte exactly once with as few
// instructions per weight as possible. The roles of a CTA live in stream.cuh.
//
// Grid: x = CTA column tiles (W consumer warps x CH 32-column tiles each) x row slices of the
// activations (16 rows each, one for M <= 16; the slice index fastest), y = CK ranks of a split
// over K (one thread-block cluster; partial tiles are sent to their owning rank over distributed
// shared memory and added in rank order: deterministic, no global scratch, no atomics).
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "internal.h"
#include "plan.h"
#include "splitk.cuh"
#include "stream.cuh"

namespace cg = cooperative_groups;

namespace w4a16 {
namespace {

using ws::Acc;
using ws::LaneRows;
using ws::WeightMaps;

// Kernel geometries: WsGeo<mode, blocks, consumer warps, tiles per warp, groups per stage,
// ring stages, groups per activation chunk, activation bytes>.
//   up to 4 rows (two-term columns): 512 or 256 columns per CTA;
//   5..8 rows and 9..16 rows (terms summed over k): 512 or 256 columns;
//   bf16 activations (one term): 512 or 256 columns.
// Compile-time knobs per form: consumer warps (_W), tiles per warp (_CH, default 16 / W), ring
// depth (_R, scaled by 16 / tiles so every form keeps 16 tiles' worth of stages in flight),
// activation chunk groups (_CG); W4A16_N2_NRING sets the narrow <= 4-row ring directly,
// W4A16_MINB caps the CTAs per SM the launch bounds ask registers for, W4A16_PDL turns on
// programmatic dependent launch. The defaults are the measured best on GB300. The wide form has
// 16 tiles (512 columns) per CTA, the narrow form 8: the same warps with half the tiles each, or
// half the warps where a fused SwiGLU warp needs its gate/up pair.
#ifndef W4A16_N2_W
#define W4A16_N2_W 4
#endif
#ifndef W4A16_N2_R
#define W4A16_N2_R 4
#endif
#ifndef W4A16_K2A_W
#define W4A16_K2A_W 4
#endif
#ifndef W4A16_K2A_R
#define W4A16_K2A_R 3
#endif
#ifndef W4A16_K2A_CG
#define W4A16_K2A_CG 8
#endif
#ifndef W4A16_K2B_W
#define W4A16_K2B_W 4
#endif
#ifndef W4A16_K2B_R
#define W4A16_K2B_R 3
#endif
#ifndef W4A16_K2B_CG
#define W4A16_K2B_CG 4
#endif
#ifndef W4A16_B16_W
#define W4A16_B16_W 4
#endif
#ifndef W4A16_B16_R
#define W4A16_B16_R 4
#endif
#ifndef W4A16_B16B_R
#define W4A16_B16B_R 3
#endif
#ifndef W4A16_B16B_CG
#define W4A16_B16B_CG 8
#endif
#ifndef W4A16_MINB
#define W4A16_MINB 2
#endif
// Launch with programmatic stream serialization (1): a launch may then overlap the tail of the
// previous kernel on its stream (only the activation loads wait for it). Off by default: the
// next grid's clusters are then placed into the slots the previous grid frees one by one, and
// when a grid needs every cluster slot of the GPU (e.g. 36 clusters of 8 CTAs) the last of its
// clusters find no room until its own CTAs exit: a second wave that costs more (up to +60 % per
// launch back to back) than the overlap saves (0.3 - 0.5 us per launch where it fits).
#ifndef W4A16_PDL
#define W4A16_PDL 0
#endif
// The narrow form is launched only when it fills the GPU this many times better than the wide;
// the <= 4-row form has its own margin (down, N = 7168: 224 wide CTAs streamed faster than 280
// narrow ones, 19.9 against 20.4 us back to back; at 16 rows the narrow ones won, 37.1 against
// 39.0 us).
#ifndef W4A16_NARROW_MARGIN
#define W4A16_NARROW_MARGIN 1.03
#endif
#ifndef W4A16_N2_NARROW_MARGIN
#define W4A16_N2_NARROW_MARGIN 1.3
#endif
// Ring depth scales with 16 / (tiles per CTA), so the narrow form keeps the wide form's bytes in
// flight per CTA.
template <int W, int CH, int R = W4A16_N2_R * 16 / (W * CH)>
using GeoN2 = ws::WsGeo<ws::kN2, 1, W, CH, 2, R, 8, 4>;
template <int W, int CH>
using GeoK2a = ws::WsGeo<ws::kK2, 1, W, CH, 2, W4A16_K2A_R * 16 / (W * CH), W4A16_K2A_CG, 4>;
template <int W, int CH>
using GeoK2b = ws::WsGeo<ws::kK2, 2, W, CH, 2, W4A16_K2B_R * 16 / (W * CH), W4A16_K2B_CG, 4>;
template <int NB, int W, int CH>
using GeoB16 = ws::WsGeo<ws::kK1, NB, W, CH, 2,
                         (NB == 1 ? W4A16_B16_R : W4A16_B16B_R) * 16 / (W * CH),
                         NB == 1 ? 8 : W4A16_B16B_CG, 2>;
#ifndef W4A16_N2_CH
#define W4A16_N2_CH (16 / W4A16_N2_W)
#endif
#ifndef W4A16_K2A_CH
#define W4A16_K2A_CH (16 / W4A16_K2A_W)
#endif
#ifndef W4A16_K2B_CH
#define W4A16_K2B_CH (16 / W4A16_K2B_W)
#endif
#ifndef W4A16_B16_CH
#define W4A16_B16_CH (16 / W4A16_B16_W)
#endif
constexpr int kN2W = W4A16_N2_W, kN2CH = W4A16_N2_CH;
constexpr int kK2aW = W4A16_K2A_W, kK2aCH = W4A16_K2A_CH;
constexpr int kK2bW = W4A16_K2B_W, kK2bCH = W4A16_K2B_CH;
constexpr int kB16W = W4A16_B16_W, kB16CH = W4A16_B16_CH;
// Resident CTAs per SM the launch bounds ask registers for: as many as fit in shared memory
// (228 KB per SM, 1 KB reserved per CTA), at most W4A16_MINB.
constexpr int fit_blocks(int smem) { return 228 * 1024 / (smem + 1024); }
template <typename L>
constexpr int min_blocks() {
  return fit_blocks(L::kAlloc) < W4A16_MINB ? (fit_blocks(L::kAlloc) < 1 ? 1 : fit_blocks(L::kAlloc))
                                            : W4A16_MINB;
}
// Split-K epilogue of geometry L: receive slots in shared memory of their own where they still
// fit as many CTAs per SM as L alone (pushes then start as soon as a rank's stream ends), else in
// the drained code ring (after a cluster barrier).
template <typename L, bool SWIGLU>
using SplitK = mma::SplitKPush<SWIGLU, L::kTiles * 32, L::MI::kRows>;
template <typename L>
constexpr int slots_off() {
  return (L::kBytes + 127) / 128 * 128;
}
template <typename L, bool SWIGLU>
constexpr bool own_slots() {
  return fit_blocks(L::kAlloc + 128 + SplitK<L, SWIGLU>::kSlotBytes) >= min_blocks<L>() &&
         L::kAlloc + 128 + SplitK<L, SWIGLU>::kSlotBytes <= 227 * 1024;
}
template <typename L, bool SWIGLU>
constexpr int smem_bytes() {
  return L::kAlloc + (own_slots<L, SWIGLU>() ? 128 + SplitK<L, SWIGLU>::kSlotBytes : 0);
}

// Output element stores: float32, or bf16 (bit pattern in uint16_t) rounded to nearest even.
__device__ __forceinline__ void store4(float* y, float4 v) { *reinterpret_cast<float4*>(y) = v; }
__device__ __forceinline__ void store4(uint16_t* y, float4 v) {
  const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
  const __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
  uint2 o;
  o.x = *reinterpret_cast<const uint32_t*>(&lo);
  o.y = *reinterpret_cast<const uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(y) = o;
}

__device__ __forceinline__ float4 swiglu4(float4 g, float4 u) {
  return make_float4(mma::silu_f(g.x) * u.x, mma::silu_f(g.y) * u.y, mma::silu_f(g.z) * u.z,
                     mma::silu_f(g.w) * u.w);
}

// Grid x = column tile x row slice (kRows rows each), the slice index fastest: the slices of a
// weight tile are resident together, so their copies of the same weight bytes meet in L2 and
// the weights come from HBM once per launch whatever M is.
struct GridPos {
  int tile, row0;
};
template <typename L>
__device__ __forceinline__ GridPos grid_pos(int M) {
  const int nz = (M + L::MI::kRows - 1) / L::MI::kRows;
  const int tile = (int)blockIdx.x / nz;
  return {tile, ((int)blockIdx.x - tile * nz) * L::MI::kRows};
}

template <typename L, bool SWIGLU, typename XT, typename YT>
__global__ void __launch_bounds__(L::kThreads, min_blocks<L>())
    ws_gemv_kernel(const __grid_constant__ WeightMaps wm, const __grid_constant__ CUtensorMap xmap,
                   YT* __restrict__ y, int M, int N, int K, unsigned int* err) {
  constexpr int MODE = L::kMode, NB = L::kNB, CH = L::kCH, G = L::kG;
  using LR = LaneRows<MODE, NB>;
  extern __shared__ __align__(1024) char smem_raw[];
  char* base = mma::align1024(smem_raw);
  cg::cluster_group cluster = cg::this_cluster();
  const int CK = (int)cluster.dim_blocks().y;
  const int rank = (int)cluster.block_index().y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const GridPos gp = grid_pos<L>(M);
  const int tile = gp.tile, xrow0 = gp.row0;
  const int Ms = min(M - xrow0, L::MI::kRows);
  const int ldy = SWIGLU ? N / 2 : N;
  y += (size_t)xrow0 * ldy;
  // This rank's groups: whole stages of G groups, split as evenly as possible.
  const int Gt = K / kGroup;
  const int U = (Gt + G - 1) / G;
  const int q0 = G * (int)((long long)rank * U / CK);
  const int q1 = min(Gt, G * (int)((long long)(rank + 1) * U / CK));
  const int nq = q1 - q0;

  ws::init_roles<L>(base);
  if (threadIdx.x == 0) ws::allow_dependents();
  __syncthreads();
  constexpr bool kOwnSlots = own_slots<L, SWIGLU>();
  if (kOwnSlots && CK > 1) mma::cluster_arrive_relaxed();  // barriers initialized, for the peers
  Acc<CH, NB> acc;
  int ex[LR::kN];
  if (warp == 0) {
    if (lane == 0) {
      ws::prefetch_tmap(&wm.codes);
      ws::prefetch_tmap(&wm.scales);
      ws::producer_loop<SWIGLU, L>(wm, base, q0, nq, tile, N, 0, err);
    }
  } else if (warp == 1) {
    if (lane == 0) ws::prefetch_tmap(&xmap);
    ws::prep_loop<XT, L>(&xmap, base, q0, nq, xrow0, err);
  } else {
    ws::consumer_loop<SWIGLU, L>(base, nq, warp - 2, err, acc, ex);
  }
  __syncthreads();  // every role is done with the rings; the code ring becomes the reduction tile

  const int w = warp - 2;
  const int h4 = 4 * mma::lane_chunk(g);
  constexpr int kT = L::kTiles;
  if (CK == 1) {
    if (warp < 2) return;
#pragma unroll
    for (int i = 0; i < LR::kN; ++i) {
      const int m = LR::row(t, i);
      if (m >= Ms) continue;
      const float f = mma::exp2i(ex[i] - 14);
      const int b = MODE == ws::kN2 ? 0 : (i >> 1), odd = i & 1;
      if constexpr (SWIGLU) {
        constexpr int H = CH / 2;
#pragma unroll
        for (int c = 0; c < H; ++c) {
          const int j = 32 * (tile * (kT / 2) + w * H + c) + h4;
          if (j < ldy)
            store4(y + (size_t)m * ldy + j,
                   swiglu4(ws::lane_result<MODE, CH, NB>(acc, c, b, odd, f),
                           ws::lane_result<MODE, CH, NB>(acc, c + H, b, odd, f)));
        }
      } else {
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const int col = 32 * (tile * kT + w * CH + c) + h4;
          if (col < N)
            store4(y + (size_t)m * N + col, ws::lane_result<MODE, CH, NB>(acc, c, b, odd, f));
        }
      }
    }
    return;
  }
  constexpr int kCols = kT * 32;
  using SK = SplitK<L, SWIGLU>;
  static_assert(kOwnSlots || SK::kSlotBytes <= L::kR * L::kCodeStage,
                "receive slots must fit in the code ring");
  const ws::Bars<L> bars(base);
  const uint32_t slots =
      ws::smem_u32(base) + (kOwnSlots ? (uint32_t)slots_off<L>() : (uint32_t)L::kCodeOff);
  if (!kOwnSlots) {
    ws::fence_proxy_async_smem();  // the ring's generic reads, before the peers' async writes
    mma::cluster_arrive();
  }
  // Own slots: every CTA of the cluster has started and initialized its receive barrier.
  // Ring slots: every CTA's ring is drained.
  mma::cluster_wait();
  const SK sk(CK, rank, slots, bars.recv);
  if (threadIdx.x == 0) ws::mbar_expect_tx(bars.recv, sk.rx_bytes(Ms));
  if (warp >= 2) {
#pragma unroll
    for (int i = 0; i < LR::kN; ++i) {
      const int m = LR::row(t, i);
      if (m >= Ms) continue;
      const float f = mma::exp2i(ex[i] - 14);
      const int b = MODE == ws::kN2 ? 0 : (i >> 1), odd = i & 1;
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        int lc;
        if constexpr (SWIGLU) {
          constexpr int H = CH / 2;
          lc = (c >= H ? kCols / 2 : 0) + 32 * (w * H + (c >= H ? c - H : c)) + h4;
        } else {
          lc = 32 * (w * CH + c) + h4;
        }
        sk.put(m, lc, ws::lane_result<MODE, CH, NB>(acc, c, b, odd, f));
      }
    }
  }
  // This rank's sends are issued. Relaxed: an owner learns that its data has landed from its
  // receive barrier (the sends' byte counts complete it with release semantics), so this arrive
  // need not wait for the stores to be performed at the peers.
  mma::cluster_arrive_relaxed();
  if (!sk.finish(Ms, tile, ldy, y) && threadIdx.x == 0)
    ws::raise_abort(reinterpret_cast<volatile int*>(base + L::kAbortOff), err);
  mma::cluster_wait();  // every peer has issued its sends: none is still to come
}

// ------------------------------------------------------------------------------ host side

template <typename L, bool SWIGLU>
int cta_tiles(int N) {
  const int tiles = SWIGLU ? ((N >> 1) + 31) / 32 : (N + 31) / 32;
  const int per = SWIGLU ? L::kTiles / 2 : L::kTiles;
  return (tiles + per - 1) / per;
}

// Weight descriptors of a [K, N] matrix for geometry L.
template <typename L, bool SWIGLU>
cudaError_t weight_maps(WeightMaps* wm, const int32_t* qw, const float* sc, int N, int K) {
  constexpr int G = L::kG, kT = L::kTiles;
  const uint64_t rows = (uint64_t)K / 8, grows = (uint64_t)K / kGroup, n = (uint64_t)N;
  const bool fast = SWIGLU ? ((N / 2) % 32 == 0) : (N % 32 == 0);
  wm->fast = fast ? 1 : 0;
  cudaError_t e;
  if (fast) {
    if (SWIGLU) {
      const uint64_t I = n / 2;
      const uint64_t dq[5] = {32, rows, I / 32, 2, 1};
      const uint64_t sq[4] = {n * 4, 128, I * 4, rows * n * 4};
      const uint32_t bq[5] = {32, 4 * G, kT / 2, 2, 1};
      e = make_tmap_nd(&wm->codes, CU_TENSOR_MAP_DATA_TYPE_INT32, CU_TENSOR_MAP_SWIZZLE_128B, qw,
                       5, dq, sq, bq);
      if (e != cudaSuccess) return e;
      const uint64_t ds[5] = {32, grows, I / 32, 2, 1};
      const uint64_t ss[4] = {n * 4, 128, I * 4, grows * n * 4};
      const uint32_t bs[5] = {32, G, kT / 2, 2, 1};
      return make_tmap_nd(&wm->scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                          CU_TENSOR_MAP_SWIZZLE_NONE, sc, 5, ds, ss, bs);
    }
    const uint64_t dq[4] = {32, rows, n / 32, 1};
    const uint64_t sq[3] = {n * 4, 128, rows * n * 4};
    const uint32_t bq[4] = {32, 4 * G, kT, 1};
    e = make_tmap_nd(&wm->codes, CU_TENSOR_MAP_DATA_TYPE_INT32, CU_TENSOR_MAP_SWIZZLE_128B, qw, 4,
                     dq, sq, bq);
    if (e != cudaSuccess) return e;
    const uint64_t ds[4] = {32, grows, n / 32, 1};
    const uint64_t ss[3] = {n * 4, 128, grows * n * 4};
    const uint32_t bs[4] = {32, G, kT, 1};
    return make_tmap_nd(&wm->scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, CU_TENSOR_MAP_SWIZZLE_NONE,
                        sc, 4, ds, ss, bs);
  }
  const uint64_t dq[3] = {n, rows, 1};
  const uint64_t sq[2] = {n * 4, rows * n * 4};
  const uint32_t bq[3] = {32, 4 * G, 1};
  e = make_tmap_nd(&wm->codes, CU_TENSOR_MAP_DATA_TYPE_INT32, CU_TENSOR_MAP_SWIZZLE_128B, qw, 3, dq,
                   sq, bq);
  if (e != cudaSuccess) return e;
  const uint64_t ds[3] = {n, grows, 1};
  const uint64_t ss[2] = {n * 4, grows * n * 4};
  const uint32_t bs[3] = {32, G, 1};
  return make_tmap_nd(&wm->scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, CU_TENSOR_MAP_SWIZZLE_NONE, sc,
                      3, ds, ss, bs);
}

// Activation descriptor: [M, K] row-major, box (32 CG inputs x kRows rows).
template <typename L, typename XT>
cudaError_t act_map(CUtensorMap* m, const XT* x, int M, int K) {
  const uint64_t d[2] = {(uint64_t)K, (uint64_t)M};
  const uint64_t s[1] = {(uint64_t)K * sizeof(XT)};
  const uint32_t b[2] = {(uint32_t)(32 * L::kCG), (uint32_t)L::MI::kRows};
  return make_tmap_nd(m,
                      sizeof(XT) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                      : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                      CU_TENSOR_MAP_SWIZZLE_NONE, x, 2, d, s, b);
}

template <typename L, bool SWIGLU, typename XT, typename YT>
struct Instance {
  static LaunchCache cache;
  static constexpr auto kernel = ws_gemv_kernel<L, SWIGLU, XT, YT>;

  static cudaError_t data(const DeviceInfo& di, const LaunchData** ld) {
    return launch_data(kernel, smem_bytes<L, SWIGLU>(), L::kThreads, cache, di, ld);
  }
  // Predicted fill of the GPU for this problem (see plan_split).
  static cudaError_t fill(int M, int N, int K, const DeviceInfo& di, double* eff) {
    const LaunchData* ld = nullptr;
    cudaError_t e = data(di, &ld);
    if (e != cudaSuccess) return e;
    const int nz = (M + L::MI::kRows - 1) / L::MI::kRows;
    const int stages = (K / kGroup + L::kG - 1) / L::kG;
    (void)plan_split(*ld, (long long)cta_tiles<L, SWIGLU>(N) * nz, stages, di, eff);
    return cudaSuccess;
  }
  static cudaError_t launch(const XT* x, const int32_t* qw, const float* sc, YT* y, int M, int N,
                            int K, const DeviceInfo& di, cudaStream_t s) {
    const LaunchData* ld = nullptr;
    cudaError_t e = data(di, &ld);
    if (e != cudaSuccess) return e;
    const int nz = (M + L::MI::kRows - 1) / L::MI::kRows;
    const int tiles = cta_tiles<L, SWIGLU>(N);
    const int stages = (K / kGroup + L::kG - 1) / L::kG;
    const int CK = plan_split(*ld, (long long)tiles * nz, stages, di, nullptr);
    WeightMaps wm;
    e = weight_maps<L, SWIGLU>(&wm, qw, sc, N, K);
    if (e != cudaSuccess) return e;
    CUtensorMap xm;
    e = act_map<L, XT>(&xm, x, M, K);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tiles * nz, CK, 1);
    cfg.blockDim = dim3(L::kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem_bytes<L, SWIGLU>();
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = CK;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = W4A16_PDL ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, wm, xm, y, M, N, K, device_error_word());
  }
};
template <typename L, bool SWIGLU, typename XT, typename YT>
LaunchCache Instance<L, SWIGLU, XT, YT>::cache;

// Of two geometries (wide: more columns per CTA, narrow: fewer), launches the wide one unless the
// narrow one fills the GPU more than `margin` times better. Wide CTAs share each activation
// fragment and each stage's fixed work between more columns.
template <typename Wide, typename Narrow, typename XT, typename YT>
cudaError_t launch_best(const XT* x, const int32_t* qw, const float* sc, YT* y, int M, int N,
                        int K, const DeviceInfo& di, cudaStream_t s,
                        double margin = W4A16_NARROW_MARGIN) {
  double ew = 0.0, en = 0.0;
  cudaError_t e = Wide::fill(M, N, K, di, &ew);
  if (e != cudaSuccess) return e;
  e = Narrow::fill(M, N, K, di, &en);
  if (e != cudaSuccess) return e;
  return ew * margin >= en ? Wide::launch(x, qw, sc, y, M, N, K, di, s)
                           : Narrow::launch(x, qw, sc, y, M, N, K, di, s);
}

// The narrow form (8 tiles per CTA) of a wide geometry with W warps of CH tiles: the same warps
// with half the tiles each, or half the warps when a fused SwiGLU warp needs its gate/up pair.
constexpr int narrow_w(int W, int CH, bool swiglu) { return CH >= (swiglu ? 4 : 2) ? W : W / 2; }
constexpr int narrow_ch(int W, int CH, bool swiglu) {
  return CH >= (swiglu ? 4 : 2) ? CH / 2 : CH;
}

template <bool SWIGLU>
cudaError_t dispatch(const float* x, const int32_t* qw, const float* sc, float* y, int M, int N,
                     int K, const DeviceInfo& di, cudaStream_t s) {
  if (M <= 4) {
    using Wide = GeoN2<kN2W, kN2CH>;
    constexpr int nw = narrow_w(kN2W, kN2CH, SWIGLU), nch = narrow_ch(kN2W, kN2CH, SWIGLU);
#ifdef W4A16_N2_NRING
    using Narrow = GeoN2<nw, nch, W4A16_N2_NRING>;
#else
    using Narrow = GeoN2<nw, nch>;
#endif
    return launch_best<Instance<Wide, SWIGLU, float, float>, Instance<Narrow, SWIGLU, float, float>>(
        x, qw, sc, y, M, N, K, di, s, W4A16_N2_NARROW_MARGIN);
  }
  if (M <= 8) {
    using Wide = GeoK2a<kK2aW, kK2aCH>;
    using Narrow = GeoK2a<narrow_w(kK2aW, kK2aCH, SWIGLU), narrow_ch(kK2aW, kK2aCH, SWIGLU)>;
    return launch_best<Instance<Wide, SWIGLU, float, float>, Instance<Narrow, SWIGLU, float, float>>(
        x, qw, sc, y, M, N, K, di, s);
  }
  using Wide = GeoK2b<kK2bW, kK2bCH>;
  using Narrow = GeoK2b<narrow_w(kK2bW, kK2bCH, SWIGLU), narrow_ch(kK2bW, kK2bCH, SWIGLU)>;
  return launch_best<Instance<Wide, SWIGLU, float, float>, Instance<Narrow, SWIGLU, float, float>>(
      x, qw, sc, y, M, N, K, di, s);
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

cudaError_t launch_gemv_b16(const uint16_t* x, const int32_t* qw, const float* sc, uint16_t* y,
                            int M, int N, int K, cudaStream_t s) {
  DeviceInfo di;
  cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return e;
  constexpr int nw = narrow_w(kB16W, kB16CH, false), nch = narrow_ch(kB16W, kB16CH, false);
  if (M <= 8)
    return launch_best<Instance<GeoB16<1, kB16W, kB16CH>, false, uint16_t, uint16_t>,
                       Instance<GeoB16<1, nw, nch>, false, uint16_t, uint16_t>>(x, qw, sc, y, M,
                                                                                N, K, di, s);
  if (M <= 16)
    return launch_best<Instance<GeoB16<2, kB16W, kB16CH>, false, uint16_t, uint16_t>,
                       Instance<GeoB16<2, nw, nch>, false, uint16_t, uint16_t>>(x, qw, sc, y, M,
                                                                                N, K, di, s);
  return cudaErrorInvalidValue;
}

}  // namespace w4a16
