// Routed-expert MoE block over INT4 experts (page "The Final Wire: How a Single Edit Integrated
// INT4 Quantization into a Native DDTree Inference Engine", section "What the Edit Actually
// Changes": the router picks top-k experts per token and each expert's gate, up and down
// projections run through the INT4 GEMM).
//
// Four launches on the caller's stream:
//   1. route    : one CTA counting-sorts the T*topk (token, slot) pairs by expert (stable, so
//                 the order inside an expert is ascending pair index) and lists active experts;
//   2. gate/up  : persistent CTAs over (active expert, tile of 8 slices = 256 gate + 256 up
//                 columns) jobs; each job streams its weight tile once for all of the expert's
//                 rows (up to 8 per pass) with the tensor-core core of mma_core.cuh and writes
//                 silu(g)*u rows of h[pairs, I] in expert-sorted order;
//   3. down     : same over (active expert, 512-column tile) of the down weights, h -> y_pair;
//   4. combine  : out[t] = sum_j topk_w[t, j] * y_pair[pos(t, j)] in slot order (the MoE block
//                 entry first runs a shared expert and starts each row from its output).
// No atomics on data, so the result is deterministic. Every weight byte of an active expert is
// read once per call (plus one more pass per further 8 rows for experts with more than 8).
#include <stdint.h>

#include "internal.h"
#include "mma_core.cuh"

namespace w4a16 {
namespace {

using namespace mma;

constexpr int kWN = 8;           // warps (64-column slices) per CTA
constexpr int kCH = 2;           // 16-byte chunks per lane per group
constexpr int kRowsPerPass = 8;  // rows of one expert per pass over a weight tile

template <int NB>
using MoeGeo = Geo<NB, kCH, kWN, 4, 24576>;

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

struct MoeLayout {
  size_t hdr, off, active, sorted, pos, h, ypair, total;
};

MoeLayout moe_layout(int T, int topk, int E, int K, int I) {
  const size_t P = (size_t)T * topk;
  MoeLayout L;
  size_t o = 0;
  L.hdr = o;    o += align256(4 * sizeof(int));
  L.off = o;    o += align256((size_t)(E + 1) * sizeof(int));
  L.active = o; o += align256((size_t)E * sizeof(int));
  L.sorted = o; o += align256(P * sizeof(int));
  L.pos = o;    o += align256(P * sizeof(int));
  L.h = o;      o += align256(P * (size_t)I * sizeof(float));
  L.ypair = o;  o += align256(P * (size_t)K * sizeof(float));
  L.total = o;
  return L;
}

// ---------------------------------------------------------------------------------- routing

__global__ void __launch_bounds__(1024) moe_route_kernel(const int32_t* __restrict__ ids, int P,
                                                         int E, int* __restrict__ hdr,
                                                         int* __restrict__ off,
                                                         int* __restrict__ active,
                                                         int* __restrict__ sorted_pair,
                                                         int* __restrict__ pair_pos,
                                                         unsigned int* err) {
  extern __shared__ int sm_int[];
  int* cnt = sm_int;         // [E]
  int* cursor = sm_int + E;  // [E]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  for (int p = tid; p < P; p += blockDim.x) {
    const int e = ids[p];
    if (e >= 0 && e < E) {
      atomicAdd(&cnt[e], 1);  // counts only: order-independent
    } else {
      pair_pos[p] = -1;
      if (err) atomicCAS(err, 0u, 1u);  // W4A16_ERR_ARG
    }
  }
  __syncthreads();
  if (tid == 0) {
    int o = 0, na = 0;
    for (int e = 0; e < E; ++e) {
      off[e] = o;
      cursor[e] = o;
      if (cnt[e] > 0) active[na++] = e;
      o += cnt[e];
    }
    off[E] = o;
    hdr[0] = na;
    hdr[1] = o;
  }
  __syncthreads();
  // Stable placement: pairs are taken in index order, warp by warp; inside a warp, lanes with
  // the same expert are ranked by lane.
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int base = 0; base < P; base += blockDim.x) {
    const int p = base + tid;
    const int e = (p < P) ? ids[p] : -1;
    const bool valid = p < P && e >= 0 && e < E;
    const int key = valid ? e : -1;
    const unsigned mask = __match_any_sync(0xffffffffu, key);
    const int rank = __popc(mask & lt_mask);
    const int leader = 31 - __clz(mask);
    for (int w = 0; w < nwarps; ++w) {
      if (warp == w) {
        int pos = 0;
        if (valid) pos = cursor[e] + rank;
        __syncwarp();
        if (valid) {
          sorted_pair[pos] = p;
          pair_pos[p] = pos;
          if (lane == leader) cursor[e] += __popc(mask);
        }
      }
      __syncthreads();
    }
  }
}

// ---------------------------------------------------------------------------------- grouped GEMV

struct GroupedArgs {
  const float* src;          // gate/up: x [T, K]; down: h [P, I]
  const int* sorted_pair;    // expert-sorted pair indices
  int topk;
  bool gather;               // gate/up: row = token of the pair; down: row = sorted position
  const int* hdr;
  const int* off;
  const int* active;
  int N;                     // columns per expert (gate/up: 2I)
  int Kr;                    // reduction length (gate/up: K; down: I)
  int tiles;
  float* dst;                // gate/up: h [P, I]; down: y_pair [P, K]
  int ldd;
  unsigned int* err;
};

template <int NB, bool SWIGLU>
__device__ __forceinline__ void grouped_pass(const GroupedArgs& a, const CUtensorMap* tq,
                                             const CUtensorMap* ts, int e, int tile, int row0,
                                             int rows, char* smem, int& seq) {
  const int warp = threadIdx.x >> 5;
  auto rowptr = [&](int m) {
    const int p = row0 + m;
    const int r = a.gather ? (a.sorted_pair[p] / a.topk) : p;
    return a.src + (size_t)r * a.Kr;
  };
  float acc[kCH][2][NB][4];
  stream_groups<NB, kCH, SWIGLU, kWN, MoeGeo<NB>>(rowptr, rows, tq, ts, e, a.N, 0,
                                                   a.Kr / kGroup, tile * kWN, smem, seq, a.err,
                                                   acc);
  store_direct<NB, kCH, SWIGLU>(acc, tile * kWN + warp, a.N, rows, a.dst + (size_t)row0 * a.ldd);
}

template <bool SWIGLU>
__global__ void __launch_bounds__(kWN * 32, 2)
    moe_grouped_kernel(const __grid_constant__ CUtensorMap tq,
                       const __grid_constant__ CUtensorMap ts, GroupedArgs a) {
  extern __shared__ __align__(1024) char smem_raw[];
  char* smem = align1024(smem_raw);
  init_barriers<MoeGeo<2>>(smem, kWN);
  int seq = 0;
  const int n_active = a.hdr[0];
  const long long total = (long long)n_active * a.tiles;
  for (long long item = blockIdx.x; item < total; item += gridDim.x) {
    const int ai = (int)(item / a.tiles);
    const int tile = (int)(item - (long long)ai * a.tiles);
    const int e = a.active[ai];
    const int r0 = a.off[e];
    const int rows = a.off[e + 1] - r0;
    for (int c0 = 0; c0 < rows; c0 += kRowsPerPass) {
      const int mr = (rows - c0) < kRowsPerPass ? (rows - c0) : kRowsPerPass;
      if (mr <= 4)
        grouped_pass<1, SWIGLU>(a, &tq, &ts, e, tile, r0 + c0, mr, smem, seq);
      else
        grouped_pass<2, SWIGLU>(a, &tq, &ts, e, tile, r0 + c0, mr, smem, seq);
    }
  }
}

// ---------------------------------------------------------------------------------- combine

// With `shared` (the shared expert's output [T, K]) each row starts from it, then adds the routed
// rows in slot order.
__global__ void moe_combine_kernel(const float* __restrict__ ypair, const int* __restrict__ pos,
                                   const float* __restrict__ w, int T, int topk, int K,
                                   const float* __restrict__ shared, float* __restrict__ out) {
  const int K4 = K >> 2;
  const long long total = (long long)T * K4;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(idx / K4);
    const int c4 = (int)(idx - (long long)t * K4);
    float4 s = shared ? reinterpret_cast<const float4*>(shared + (size_t)t * K)[c4]
                      : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < topk; ++j) {
      const int p = pos[t * topk + j];
      if (p < 0) continue;
      const float wt = w[t * topk + j];
      const float4 v = reinterpret_cast<const float4*>(ypair + (size_t)p * K)[c4];
      s.x = fmaf(wt, v.x, s.x);
      s.y = fmaf(wt, v.y, s.y);
      s.z = fmaf(wt, v.z, s.z);
      s.w = fmaf(wt, v.w, s.w);
    }
    reinterpret_cast<float4*>(out + (size_t)t * K)[c4] = s;
  }
}

__global__ void topk_softmax_kernel(const float* __restrict__ logits, float* __restrict__ weights,
                                    int T, int topk) {
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x) {
    const float* l = logits + (size_t)t * topk;
    float mx = l[0];
    for (int j = 1; j < topk; ++j) mx = fmaxf(mx, l[j]);
    float ex[32];
    float sum = 0.0f;
    for (int j = 0; j < topk; ++j) {
      ex[j] = expf(l[j] - mx);
      sum += ex[j];
    }
    for (int j = 0; j < topk; ++j) weights[(size_t)t * topk + j] = ex[j] / sum;
  }
}

// Both NB paths of the grouped kernel share one shared-memory buffer (the larger layout); the
// rings and barriers sit at the same offsets in both.
static_assert(MoeGeo<1>::kBarOff == MoeGeo<2>::kBarOff, "shared barrier offset");
constexpr int kMoeSmem =
    MoeGeo<2>::kAlloc > MoeGeo<1>::kAlloc ? MoeGeo<2>::kAlloc : MoeGeo<1>::kAlloc;

template <bool SWIGLU>
cudaError_t launch_grouped(const GroupedArgs& a, const int32_t* qw, const float* sc, int E,
                           const DeviceInfo& di, cudaStream_t s) {
  static PerDeviceOnce<int> occ_cache;  // resident CTAs per SM
  auto kern = moe_grouped_kernel<SWIGLU>;
  const int* occ = nullptr;
  cudaError_t e = occ_cache.get(di.device, [&](int& o) {
    cudaError_t r =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMoeSmem);
    if (r != cudaSuccess) return r;
    int n = 0;
    r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kWN * 32, kMoeSmem);
    if (r != cudaSuccess) return r;
    o = n < 1 ? 1 : n;
    return cudaSuccess;
  }, &occ);
  if (e != cudaSuccess) return e;
  CUtensorMap tq, ts;
  e = make_tmap(&tq, 0, qw, (uint64_t)a.N, (uint64_t)(a.Kr / 8), (uint64_t)E, 32,
                            kRows);
  if (e != cudaSuccess) return e;
  e = make_tmap(&ts, 1, sc, (uint64_t)a.N, (uint64_t)(a.Kr / kGroup), (uint64_t)E, 32,
                kRows / 4);
  if (e != cudaSuccess) return e;
  kern<<<di.sm_count * *occ, kWN * 32, kMoeSmem, s>>>(tq, ts, a);
  return cudaGetLastError();
}

}  // namespace

size_t moe_workspace_size(int T, int topk, int E, int K, int I) {
  return moe_layout(T, topk, E, K, I).total;
}

size_t moe_block_workspace_size(int T, int topk, int E, int K, int I, int Is) {
  return moe_layout(T, topk, E, K, I).total + align256((size_t)T * Is * sizeof(float)) +
         align256((size_t)T * K * sizeof(float));
}

cudaError_t launch_moe(const float* x, const int32_t* ids, const float* w, int T, int topk, int E,
                       const int32_t* qw_gu, const float* sc_gu, const int32_t* qw_dn,
                       const float* sc_dn, float* out, int K, int I, void* ws, size_t ws_bytes,
                       cudaStream_t s) {
  return launch_moe_block(x, ids, w, T, topk, E, qw_gu, sc_gu, qw_dn, sc_dn, nullptr, nullptr,
                          nullptr, nullptr, 0, out, K, I, ws, ws_bytes, s);
}

// The routed experts as in launch_moe, plus (when qs_gu is given) a shared expert that every
// token goes through with weight 1: its gate/up + SwiGLU and down projections run as dense
// small-M GEMMs (one launch each, 16-row slices as grid z) into the workspace, and the combine
// starts each row from it.
cudaError_t launch_moe_block(const float* x, const int32_t* ids, const float* w, int T, int topk,
                             int E, const int32_t* qw_gu, const float* sc_gu,
                             const int32_t* qw_dn, const float* sc_dn, const int32_t* qs_gu,
                             const float* ss_gu, const int32_t* qs_dn, const float* ss_dn, int Is,
                             float* out, int K, int I, void* ws, size_t ws_bytes,
                             cudaStream_t s) {
  (void)ws_bytes;
  DeviceInfo di;
  cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return e;
  const MoeLayout L = moe_layout(T, topk, E, K, I);
  char* base = static_cast<char*>(ws);
  int* hdr = reinterpret_cast<int*>(base + L.hdr);
  int* off = reinterpret_cast<int*>(base + L.off);
  int* active = reinterpret_cast<int*>(base + L.active);
  int* sorted = reinterpret_cast<int*>(base + L.sorted);
  int* pos = reinterpret_cast<int*>(base + L.pos);
  float* h = reinterpret_cast<float*>(base + L.h);
  float* ypair = reinterpret_cast<float*>(base + L.ypair);
  const int P = T * topk;

  moe_route_kernel<<<1, 1024, 2 * (size_t)E * sizeof(int), s>>>(ids, P, E, hdr, off, active,
                                                                sorted, pos,
                                                                device_error_word());
  if ((e = cudaGetLastError()) != cudaSuccess) return e;

  GroupedArgs gu;
  gu.src = x;
  gu.sorted_pair = sorted;
  gu.topk = topk;
  gu.gather = true;
  gu.hdr = hdr;
  gu.off = off;
  gu.active = active;
  gu.err = device_error_word();
  gu.N = 2 * I;
  gu.Kr = K;
  gu.tiles = ((I + 16 * kCH - 1) / (16 * kCH) + kWN - 1) / kWN;
  gu.dst = h;
  gu.ldd = I;
  if ((e = launch_grouped<true>(gu, qw_gu, sc_gu, E, di, s)) != cudaSuccess) return e;

  GroupedArgs dn = gu;
  dn.src = h;
  dn.gather = false;
  dn.N = K;
  dn.Kr = I;
  dn.tiles = ((K + 32 * kCH - 1) / (32 * kCH) + kWN - 1) / kWN;
  dn.dst = ypair;
  dn.ldd = K;
  if ((e = launch_grouped<false>(dn, qw_dn, sc_dn, E, di, s)) != cudaSuccess) return e;

  float* ys = nullptr;
  if (qs_gu) {
    float* hs = reinterpret_cast<float*>(base + L.total);
    ys = reinterpret_cast<float*>(base + L.total + align256((size_t)T * Is * sizeof(float)));
    for (int m0 = 0; m0 < T; m0 += kGemvMaxRowsPerLaunch) {
      const int mc = T - m0 < kGemvMaxRowsPerLaunch ? T - m0 : kGemvMaxRowsPerLaunch;
      if ((e = launch_gemv(x + (size_t)m0 * K, qs_gu, ss_gu, hs + (size_t)m0 * Is, mc, 2 * Is, K,
                           true, s)) != cudaSuccess)
        return e;
      if ((e = launch_gemv(hs + (size_t)m0 * Is, qs_dn, ss_dn, ys + (size_t)m0 * K, mc, K, Is,
                           false, s)) != cudaSuccess)
        return e;
    }
  }

  const long long total4 = (long long)T * (K / 4);
  long long blocks = (total4 + 255) / 256;
  if (blocks > (long long)di.sm_count * 16) blocks = (long long)di.sm_count * 16;
  moe_combine_kernel<<<(int)(blocks < 1 ? 1 : blocks), 256, 0, s>>>(ypair, pos, w, T, topk, K,
                                                                    ys, out);
  return cudaGetLastError();
}

cudaError_t launch_topk_softmax(const float* logits, float* weights, int T, int topk,
                                cudaStream_t s) {
  const int blocks = (T + 127) / 128;
  topk_softmax_kernel<<<blocks, 128, 0, s>>>(logits, weights, T, topk);
  return cudaGetLastError();
}

}  // namespace w4a16
