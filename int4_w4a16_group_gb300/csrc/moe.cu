// Routed-expert MoE block over INT4 experts (page "The Final Wire: How a Single Edit Integrated
// INT4 Quantization into a Native DDTree Inference Engine", section "What the Edit Actually
// Changes": the router picks top-k experts per token and each expert's gate, up and down
// projections run through the INT4 GEMM).
//
// Four launches on the caller's stream:
//   1. route    : one CTA counting-sorts the T*topk (token, slot) pairs by expert (stable, so
//                 the order inside an expert is ascending pair index) and lists active experts;
//   2. gate/up  : persistent CTAs (two per SM) on the warp-specialized streaming core of
//                 stream.cuh walk items (active expert, tile of 256 gate + 256 up columns),
//                 CTA b taking items b, b + grid, ...; an item is one job per pass of up to 4
//                 of the expert's rows (gathered with one-row TMA boxes), and each job streams
//                 the item's weights once and writes silu(g)*u rows of h[pairs, I] in
//                 expert-sorted order;
//   3. down     : same over (active expert, 512-column tile) of the down weights, h -> y_pair;
//   4. combine  : out[t] = sum_j topk_w[t, j] * y_pair[pos(t, j)] in slot order (the MoE block
//                 entry first runs a shared expert and starts each row from its output).
// No atomics on data, so the result is deterministic. Every weight byte of an active expert is
// read once per pass of 4 rows (experts average 1.8 rows in the T = 64, top-8 workload).
#include <stdint.h>

#include "internal.h"
#include "stream.cuh"

namespace w4a16 {
namespace {

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
//
// Persistent warp-specialized CTAs (stream.cuh roles) walk jobs (active expert, 512-column
// tile [gate/up: 256 gate + the matching 256 up columns], pass of up to 4 of the expert's rows):
// each job streams its tile of the expert's packed weights once (TMA boxes with the expert as
// the outermost coordinate) and accumulates the pass's rows in the two-term-column mode. The
// prep warp gathers the pass's rows (one-row TMA boxes; rows past the pass read as zero). The
// ring, chunk and barrier phases run on across jobs, so a CTA's next job streams while its last
// one stores.

using MoeL = ws::WsGeo<ws::kN2, 1, 4, 4, 2, 4, 8, 4>;
constexpr int kPassRows = 4;

struct GroupedArgs {
  const int* sorted_pair;    // expert-sorted pair indices
  int topk;
  bool gather;               // gate/up: source row = token of the pair; down: the sorted position
  int src_rows;              // rows of the source (gate/up: T; down: P)
  const int* hdr;
  const int* off;
  const int* active;
  int N;                     // columns per expert (gate/up: 2I)
  int Kr;                    // reduction length (gate/up: K; down: I)
  int tiles;                 // 512-column tiles per expert
  float* dst;                // gate/up: h [P, I]; down: y_pair [P, K]
  int ldd;
  unsigned int* err;
};

// Job cursor: (active expert index, tile, pass) in the order every role of a CTA walks them.
struct JobCursor {
  long long item;  // active expert index * tiles + tile
  int pass;
  __device__ __forceinline__ JobCursor(long long start) : item(start), pass(0) {}
  // Fills the job; returns false past the end.
  __device__ __forceinline__ bool get(const GroupedArgs& a, int n_active, int* e, int* tile,
                                      int* r0, int* rows) const {
    if (item >= (long long)n_active * a.tiles) return false;
    const int ai = (int)(item / a.tiles);
    *tile = (int)(item - (long long)ai * a.tiles);
    *e = a.active[ai];
    const int o0 = a.off[*e], o1 = a.off[*e + 1];
    *r0 = o0 + kPassRows * pass;
    *rows = min(kPassRows, o1 - *r0);
    return true;
  }
  __device__ __forceinline__ void next(const GroupedArgs& a, int rows_total) {
    if (kPassRows * (pass + 1) < rows_total) {
      ++pass;
    } else {
      pass = 0;
      item += gridDim.x;
    }
  }
};

__device__ __forceinline__ int expert_rows(const GroupedArgs& a, int e) {
  return a.off[e + 1] - a.off[e];
}

template <bool SWIGLU>
__device__ __forceinline__ void moe_producer(const ws::WeightMaps& wm, char* base,
                                             const GroupedArgs& a, int n_active) {
  using L = MoeL;
  constexpr int R = L::kR, G = L::kG;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + L::kAbortOff);
  const ws::Bars<L> bars(base);
  const uint32_t codes = ws::smem_u32(base + L::kCodeOff);
  const uint32_t scales = ws::smem_u32(base + L::kScaleOff);
  const int nst = (a.Kr / kGroup + G - 1) / G;
  int st = 0;
  uint32_t ph = 0;
  long long issued = 0;
  bool ok = true;
  JobCursor jc(blockIdx.x);
  int e, tile, r0, rows;
  while (ok && jc.get(a, n_active, &e, &tile, &r0, &rows)) {
    for (int s = 0; s < nst; ++s) {
      if (issued >= R && !ws::wait_phase(bars.empty + 8 * st, ph ^ 1, abort_flag)) {
        ws::raise_abort(abort_flag, a.err);
        ok = false;
        break;
      }
      ws::issue_stage<L::kW, L::kCH, G, SWIGLU, L>(wm, codes + st * L::kCodeStage,
                                                    scales + st * L::kScaleStage,
                                                    bars.full + 8 * st, s * G, tile, a.N, e);
      ++issued;
      if (++st == R) {
        st = 0;
        ph ^= 1;
      }
    }
    jc.next(a, expert_rows(a, e));
  }
  for (long long s = issued > R ? issued - R : 0; s < issued; ++s)
    (void)mma::mbar_wait(bars.full + 8 * (int)(s % R), (uint32_t)((s / R) & 1),
                         ws::kWaitLimitNs / 16);
}

// Issues the raw rows of one chunk (lane 0): row m < rows is source row src(r0 + m), the others
// are read past the end of the source (zeros).
__device__ __forceinline__ void moe_issue_chunk(const CUtensorMap* xmap, const GroupedArgs& a,
                                                uint32_t dst, uint32_t bar, int k0, int r0,
                                                int rows) {
  using L = MoeL;
  ws::mbar_expect_tx(bar, L::kXRawBytes);
  for (int m = 0; m < kPassRows; ++m) {
    int src = a.src_rows;
    if (m < rows) src = a.gather ? a.sorted_pair[r0 + m] / a.topk : r0 + m;
    ws::tma_load_2d(dst + m * (L::kXRawBytes / kPassRows), xmap, k0, src, bar);
  }
}

__device__ __forceinline__ void moe_prep(const CUtensorMap* xmap, char* base, const GroupedArgs& a,
                                         int n_active) {
  using L = MoeL;
  constexpr int CG = L::kCG;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + L::kAbortOff);
  const ws::Bars<L> bars(base);
  const uint32_t xraw = ws::smem_u32(base + L::kXRawOff);
  const int Gt = a.Kr / kGroup;
  const int nch = (Gt + CG - 1) / CG;  // chunks per job
  // Issue cursor (lane 0): job and chunk of the next raw chunk to load.
  JobCursor ic(blockIdx.x);
  int ic_chunk = 0;
  long long issued = 0;
  auto issue_next = [&](int buf) {  // lane 0; returns nothing, advances the cursor
    int e, tile, r0, rows;
    if (!ic.get(a, n_active, &e, &tile, &r0, &rows)) return;
    moe_issue_chunk(xmap, a, xraw + buf * L::kXRawBytes, bars.xfull + 8 * buf,
                    32 * CG * ic_chunk, r0, rows);
    ++issued;
    if (++ic_chunk == nch) {
      ic_chunk = 0;
      ic.next(a, expert_rows(a, e));
    }
  };
  if (lane == 0) {
    issue_next(0);
    issue_next(1);
  }
  long long c = 0;  // chunks converted so far
  int eprev[1] = {0};
  bool ok = true;
  JobCursor jc(blockIdx.x);
  int e, tile, r0, rows;
  while (ok && jc.get(a, n_active, &e, &tile, &r0, &rows)) {
    for (int cj = 0; cj < nch; ++cj, ++c) {
      const int b = (int)(c & 1);
      const uint32_t par = (uint32_t)((c >> 1) & 1);
      bool good = ws::wait_phase(bars.xfull + 8 * b, par, abort_flag);
      if (good && c >= 2) good = ws::wait_phase(bars.fempty + 8 * b, par ^ 1, abort_flag);
      if (!__all_sync(0xffffffffu, good)) {
        if (lane == 0) ws::raise_abort(abort_flag, a.err);
        ok = false;
        break;
      }
      const int ngr = Gt - cj * CG < CG ? Gt - cj * CG : CG;
      ws::prep_chunk<ws::kN2, 1, float, L>(base, b, ngr, eprev, cj == 0);
      ws::mbar_arrive(bars.ffull + 8 * b);
      ws::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) issue_next(b);
    }
    jc.next(a, expert_rows(a, e));
  }
  if (lane == 0) {
    for (long long i = issued > 2 ? issued - 2 : 0; i < issued; ++i)
      (void)mma::mbar_wait(bars.xfull + 8 * (int)(i & 1), (uint32_t)((i >> 1) & 1),
                           ws::kWaitLimitNs / 16);
  }
}

template <bool SWIGLU>
__device__ __forceinline__ void moe_consumers(char* base, const GroupedArgs& a, int n_active) {
  using L = MoeL;
  constexpr int CH = L::kCH, G = L::kG, R = L::kR, CG = L::kCG, W = L::kW;
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3, w = (threadIdx.x >> 5) - 2;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + L::kAbortOff);
  const ws::Bars<L> bars(base);
  const int h = mma::lane_chunk(g);
  const uint32_t codes = ws::smem_u32(base + L::kCodeOff);
  const uint32_t scales = ws::smem_u32(base + L::kScaleOff) + h * 16;
  const uint32_t frag = ws::smem_u32(base + L::kFragOff) + lane * 16;
  const int* fexp = reinterpret_cast<const int*>(base + L::kExpOff);
  const int Gt = a.Kr / kGroup;
  const int nch = (Gt + CG - 1) / CG;
  int st = 0;
  uint32_t ph = 0;
  long long c = 0;
  bool ok = true;
  JobCursor jc(blockIdx.x);
  int e, tile, r0, rows;
  while (ok && jc.get(a, n_active, &e, &tile, &r0, &rows)) {
    ws::Acc<CH, 1> acc;
#pragma unroll
    for (int cc = 0; cc < CH; ++cc)
#pragma unroll
      for (int T = 0; T < 2; ++T)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc.v[cc][T][0][r] = 0.0f;
    int ex = 0;
    for (int cj = 0; cj < nch && ok; ++cj, ++c) {
      const int b = (int)(c & 1);
      ok = ws::wait_phase(bars.ffull + 8 * b, (uint32_t)((c >> 1) & 1), abort_flag);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      const bool changed = cj == 0 || fexp[L::kExpInts * b + L::kExpFlag] != 0;
      const int en = changed ? fexp[L::kExpInts * b + t] : ex;
      if (cj > 0 && changed) {
        const int d = ex - en;
        const float f = mma::exp2i(d >> 1) * mma::exp2i(d - (d >> 1));
#pragma unroll
        for (int cc = 0; cc < CH; ++cc)
#pragma unroll
          for (int T = 0; T < 2; ++T)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc.v[cc][T][0][r] *= f;
      }
      ex = en;
      const int ngr = Gt - cj * CG < CG ? Gt - cj * CG : CG;
      const uint32_t fr = frag + b * L::kFragBytes;
      for (int q = 0; q < ngr; q += G) {
        if (!ws::wait_phase(bars.full + 8 * st, ph, abort_flag)) ok = false;
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        const uint32_t cs = codes + st * L::kCodeStage, ss = scales + st * L::kScaleStage;
#pragma unroll(ws::kGroupUnroll)
        for (int j = 0; j < G; ++j)
          if (q + j < ngr)
            ws::consume_group<ws::kN2, 1, W, CH, SWIGLU, L>(cs + ws::code_offset(j, t, h),
                                                            ss + j * 128,
                                                            fr + (q + j) * 512, w, acc);
        __syncwarp();
        if (lane == 0) ws::mbar_arrive(bars.empty + 8 * st);
        if (++st == R) {
          st = 0;
          ph ^= 1;
        }
      }
      __syncwarp();
      if (ok && lane == 0) ws::mbar_arrive(bars.fempty + 8 * b);
    }
    if (!ok) break;
    // lane row t of the pass -> destination row r0 + t
    if (t < rows) {
      const float f = mma::exp2i(ex - 14);
      float* dst = a.dst + (size_t)(r0 + t) * a.ldd;
      const int h4 = 4 * h;
      if constexpr (SWIGLU) {
        constexpr int H = CH / 2, TT = L::kTiles / 2;
#pragma unroll
        for (int cc = 0; cc < H; ++cc) {
          const int j = 32 * (tile * TT + w * H + cc) + h4;
          const float4 gv = ws::lane_result<ws::kN2, CH, 1>(acc, cc, 0, 0, f);
          const float4 uv = ws::lane_result<ws::kN2, CH, 1>(acc, cc + H, 0, 0, f);
          if (j < (a.N >> 1))
            *reinterpret_cast<float4*>(dst + j) =
                make_float4(mma::silu_f(gv.x) * uv.x, mma::silu_f(gv.y) * uv.y,
                            mma::silu_f(gv.z) * uv.z, mma::silu_f(gv.w) * uv.w);
        }
      } else {
#pragma unroll
        for (int cc = 0; cc < CH; ++cc) {
          const int col = 32 * (tile * L::kTiles + w * CH + cc) + h4;
          if (col < a.N)
            *reinterpret_cast<float4*>(dst + col) =
                ws::lane_result<ws::kN2, CH, 1>(acc, cc, 0, 0, f);
        }
      }
    }
    jc.next(a, expert_rows(a, e));
  }
  if (!ok && lane == 0) ws::raise_abort(abort_flag, a.err);
}

template <bool SWIGLU>
__global__ void __launch_bounds__(MoeL::kThreads, 2)
    moe_grouped_kernel(const __grid_constant__ ws::WeightMaps wm,
                       const __grid_constant__ CUtensorMap xmap, GroupedArgs a) {
  extern __shared__ __align__(1024) char smem_raw[];
  char* base = mma::align1024(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_active = a.hdr[0];
  ws::init_roles<MoeL>(base);
  __syncthreads();
  if (warp == 0) {
    if (lane == 0) moe_producer<SWIGLU>(wm, base, a, n_active);
  } else if (warp == 1) {
    moe_prep(&xmap, base, a, n_active);
  } else {
    moe_consumers<SWIGLU>(base, a, n_active);
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

template <bool SWIGLU>
cudaError_t launch_grouped(const GroupedArgs& a, const float* src, const int32_t* qw,
                           const float* sc, int E, const DeviceInfo& di, cudaStream_t s) {
  using L = MoeL;
  static PerDeviceOnce<int> occ_cache;  // resident CTAs per SM
  auto kern = moe_grouped_kernel<SWIGLU>;
  const int* occ = nullptr;
  cudaError_t e = occ_cache.get(di.device, [&](int& o) {
    cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L::kAlloc);
    if (r != cudaSuccess) return r;
    int n = 0;
    r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, L::kThreads, L::kAlloc);
    if (r != cudaSuccess) return r;
    o = n < 1 ? 1 : n;
    return cudaSuccess;
  }, &occ);
  if (e != cudaSuccess) return e;
  // Weights [E][Kr/8][N] / [E][Kr/32][N]: columns x rows x 32-column tiles [x gate/up half]
  // x expert, boxes of one stage of a CTA's tiles.
  ws::WeightMaps wm;
  wm.fast = 1;
  const uint64_t n = (uint64_t)a.N, rows = (uint64_t)a.Kr / 8, grows = (uint64_t)a.Kr / kGroup;
  const uint64_t ne = (uint64_t)E;
  if (SWIGLU) {
    const uint64_t I = n / 2;
    const uint64_t dq[5] = {32, rows, I / 32, 2, ne}, sq[4] = {n * 4, 128, I * 4, rows * n * 4};
    const uint32_t bq[5] = {32, 4 * L::kG, L::kTiles / 2, 2, 1};
    e = make_tmap_nd(&wm.codes, CU_TENSOR_MAP_DATA_TYPE_INT32, CU_TENSOR_MAP_SWIZZLE_128B, qw, 5,
                     dq, sq, bq);
    if (e != cudaSuccess) return e;
    const uint64_t ds[5] = {32, grows, I / 32, 2, ne}, ss[4] = {n * 4, 128, I * 4, grows * n * 4};
    const uint32_t bs[5] = {32, L::kG, L::kTiles / 2, 2, 1};
    e = make_tmap_nd(&wm.scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, CU_TENSOR_MAP_SWIZZLE_NONE, sc,
                     5, ds, ss, bs);
  } else {
    const uint64_t dq[4] = {32, rows, n / 32, ne}, sq[3] = {n * 4, 128, rows * n * 4};
    const uint32_t bq[4] = {32, 4 * L::kG, L::kTiles, 1};
    e = make_tmap_nd(&wm.codes, CU_TENSOR_MAP_DATA_TYPE_INT32, CU_TENSOR_MAP_SWIZZLE_128B, qw, 4,
                     dq, sq, bq);
    if (e != cudaSuccess) return e;
    const uint64_t ds[4] = {32, grows, n / 32, ne}, ss[3] = {n * 4, 128, grows * n * 4};
    const uint32_t bs[4] = {32, L::kG, L::kTiles, 1};
    e = make_tmap_nd(&wm.scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, CU_TENSOR_MAP_SWIZZLE_NONE, sc,
                     4, ds, ss, bs);
  }
  if (e != cudaSuccess) return e;
  // Source rows [src_rows][Kr], one row per box (the prep warp gathers a pass's rows).
  CUtensorMap xm;
  const uint64_t dx[2] = {(uint64_t)a.Kr, (uint64_t)a.src_rows}, sx[1] = {(uint64_t)a.Kr * 4};
  const uint32_t bx[2] = {32 * L::kCG, 1};
  e = make_tmap_nd(&xm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, CU_TENSOR_MAP_SWIZZLE_NONE, src, 2, dx,
                   sx, bx);
  if (e != cudaSuccess) return e;
  kern<<<di.sm_count * *occ, L::kThreads, L::kAlloc, s>>>(wm, xm, a);
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
// small-M GEMMs (one launch each, all 16-row slices in its grid) into the workspace, and the combine
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
  gu.sorted_pair = sorted;
  gu.topk = topk;
  gu.gather = true;
  gu.src_rows = T;
  gu.hdr = hdr;
  gu.off = off;
  gu.active = active;
  gu.err = device_error_word();
  gu.N = 2 * I;
  gu.Kr = K;
  gu.tiles = (I + 16 * MoeL::kTiles - 1) / (16 * MoeL::kTiles);
  gu.dst = h;
  gu.ldd = I;
  if ((e = launch_grouped<true>(gu, x, qw_gu, sc_gu, E, di, s)) != cudaSuccess) return e;

  GroupedArgs dn = gu;
  dn.gather = false;
  dn.src_rows = P;
  dn.N = K;
  dn.Kr = I;
  dn.tiles = (K + 32 * MoeL::kTiles - 1) / (32 * MoeL::kTiles);
  dn.dst = ypair;
  dn.ldd = K;
  if ((e = launch_grouped<false>(dn, h, qw_dn, sc_dn, E, di, s)) != cudaSuccess) return e;

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
