// Large-M (prefill) contraction on the 5th-generation tensor cores (tcgen05, TMEM, TMA):
//   y[M, N] (bf16) = x[M, K] (bf16) @ bf16(dequant(qw, sc)) with float32 accumulation.
// The pages' activations are float32 and their kernel has no large-M form; this path serves
// batched prefill, where the op really is a dense contraction.
//
// Two CTAs of a cluster (on two SMs) share each MMA (cta_group::2). The MMA runs transposed:
// A (M = 256) = 256 dequantized weight columns, 128 in each CTA's shared memory; B (N = tm <=
// 256) = tm activation rows, tm/2 in each CTA; each CTA's TMEM holds D for its 128 columns x
// tm rows. Against one CTA per tile this halves, per SM, the x bytes TMA brings in, the operand
// bytes the tensor core reads from shared memory and the MMA instructions issued, and a ring
// stage shrinks to 37 KB so six fit. Persistent pairs walk tiles of 256 columns x tm rows, row
// blocks fastest, so a weight block's codes are reused from L2 while x stays L2-resident.
//
// Each CTA has one ring of stages, each holding what one 64-deep K block needs: the dequantized
// bf16 weight tile (128 x 64, 16 KB), the CTA's half of the x tile (tm/2 x 64 bf16), 8 packed rows
// x 128 columns of codes and 2 rows of scales. Each hand-off is one barrier, and each barrier's
// completion implies the earlier ones:
//   * a TMA producer warp (per CTA) waits until the MMAs of the stage's previous use have
//     completed (consumed, signalled to both CTAs by the MMA commit), then loads x (128-byte
//     swizzle = the UMMA K-major canonical layout), codes and scales (full);
//   * 8 dequant warps per CTA (two threads per weight column, one per scale group of the k-block)
//     wait for full and turn each packed word (8 consecutive k of one column) into 8 bf16 values:
//     ((w >> 4j) & 0x000F000F) | 0x43004300 is the bf16 pair (128 + n_j, 128 + n_{j+4}); a bf16
//     FMA subtracts 136 exactly, another multiplies by the bf16 group scale; byte permutes
//     restore k order; one 16-byte store per word writes the swizzled K-major weight tile. Then
//     they arrive on the even CTA's wready, or, in the odd CTA, on a local barrier that one relay
//     thread forwards: it releases the CTA's shared-memory writes at cluster scope (the
//     shared-memory-restricted fence) and arrives remotely on wready (a full cluster-scope
//     release costs about a microsecond, and even the restricted one is cheaper paid once per
//     stage than by each of 8 warps);
//   * one thread of the even CTA waits for wready alone (it follows both CTAs' full, which follow
//     consumed), issues 4 pair MMAs (M = 256, N = tm, K = 16, bf16 x bf16 -> f32) into a TMEM
//     accumulator and commits once to consumed in both CTAs;
//   * 4 epilogue warps per CTA drain the finished accumulator (double-buffered, 2 x 256 TMEM
//     columns): lane = weight column, so each 32-row tcgen05.ld gives a lane 32 rows of its
//     column, stored as bf16 (consecutive lanes write consecutive columns of a row); then they
//     arrive on the even CTA's accempty.
// Every barrier wait is bounded; a timeout sets the device error word and the CTA winds down.
#include <cuda_bf16.h>

#include "internal.h"
#include "mma_core.cuh"
#include "tc_core.cuh"

namespace w4a16 {
namespace {

using namespace mma;

// Hand-offs recur every few hundred nanoseconds: poll, do not sleep.
#define PF_WAIT mbar_wait_poll

constexpr int TN = 128;  // weight columns per CTA (256 per pair = the MMA's M)
constexpr int TM = 256;  // activation rows per tile at most = MMA N (half in each CTA)
constexpr int BK = 64;
// Shared memory for the ring, all but the barriers of the 227 KB a CTA may use; as many stages as
// fit are used (6 at tm = 256, up to kMaxStages for small tm). The ring round trip (TMA latency,
// dequant, the relay, the MMAs) spans several stages, so each one counts: 5 stages ran at
// 1550 TFLOP/s, 6 at 1617 (M = 4096).
#ifndef W4A16_PREFILL_RING_KB
#define W4A16_PREFILL_RING_KB 222
#endif
constexpr int kRingBytes = W4A16_PREFILL_RING_KB * 1024;
constexpr int kMaxStages = 8;
constexpr int kEpiWarps = 4;  // warps 0..3 (TMEM lane quadrants 0..3)
constexpr int kProdWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kDeqWarp0 = 6;
constexpr int kDeqWarps = 2 * TN / 32;  // two threads per weight column
constexpr int kRelayWarp = kDeqWarp0 + kDeqWarps;  // odd CTA: forwards dequant completion
constexpr int kThreads = (kRelayWarp + 1) * 32;
constexpr int kAccCols = TM;
constexpr int kTmemCols = 2 * kAccCols;

constexpr int kWBytes = TN * BK * 2;
constexpr int kQBytes = (BK / 8) * TN * 4;
constexpr int kSBytes = (BK / 32) * TN * 4;
constexpr int kBarOff = kRingBytes;
// barriers: full[8] | wready[8] | consumed[8] | pready[8] | accfull[2] | accempty[2] | drain
// (wready, accempty and drain are used in the even CTA only, pready in the odd CTA only)
constexpr int kFull = 0, kWReady = kMaxStages, kConsumed = 2 * kMaxStages,
              kPReady = 3 * kMaxStages, kAccFull = 4 * kMaxStages, kAccEmpty = kAccFull + 2,
              kDrain = kAccEmpty + 2;
constexpr int kNumBars = kDrain + 1;
constexpr int kMiscOff = kBarOff + kNumBars * 8;  // [0] TMEM base, [1] abort flag
constexpr int kSmemBytes = kMiscOff + 16;
constexpr int kSmemAlloc = kSmemBytes + 1024;
// Instruction descriptor: bf16 x bf16 -> f32, M = 256 (the pair), both operands K-major; N (the
// tile's row count) is added at run time.
constexpr uint32_t kIdescNoN = tc::idesc_f16(true, 2 * TN, 0);
static_assert(kRingBytes >= 6 * (kWBytes + TM / 2 * BK * 2 + kQBytes + kSBytes),
              "six full-width stages");
static_assert(kSmemAlloc <= 227 * 1024, "shared memory per CTA");
static_assert(kTmemCols <= 512, "TMEM columns per SM");

__device__ __forceinline__ uint32_t bf16x2_fma(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;\n" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;\n" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
__device__ __forceinline__ uint32_t lop_and_or_bf(uint32_t a, uint32_t mask) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;\n" : "=r"(r) : "r"(a), "r"(mask), "r"(0x43004300u));
  return r;
}

// One packed word (k = 8i .. 8i+7 of a column) times its bf16 scale pair -> 8 bf16 in k order.
__device__ __forceinline__ uint4 dequant_word_bf16(uint32_t w, uint32_t s2) {
  const uint32_t ONE = 0x3F803F80u;    // (1, 1)
  const uint32_t M136 = 0xC308C308u;   // (-136, -136)
  const uint32_t NEG0 = 0x80008000u;  // (-0, -0)
  uint32_t v[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t p = lop_and_or_bf(w >> (4 * j), 0x000F000Fu);  // (128 + n_j, 128 + n_{j+4})
    v[j] = bf16x2_fma(bf16x2_fma(p, ONE, M136), s2, NEG0);      // (n - 8) * s, k = j, j + 4
  }
  uint4 o;
  o.x = prmt(v[0], v[1], 0x5410u);  // k 0, 1
  o.y = prmt(v[2], v[3], 0x5410u);  // k 2, 3
  o.z = prmt(v[0], v[1], 0x7632u);  // k 4, 5
  o.w = prmt(v[2], v[3], 0x7632u);  // k 6, 7
  return o;
}

// Position in a ring of n stages: stage index and the parity of its current use (no division
// on the issue path).
struct RingPos {
  int s = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void next(int n) {
    if (++s == n) {
      s = 0;
      ph ^= 1u;
    }
  }
};

// Pair tile t: weight columns nb*256 .. +255 (CTA rank r holds nb*256 + 128 r ..) and
// activation rows mb*tm .. +tm-1 (rank r holds mb*tm + r*tm/2 ..), mb = t % mblocks.
__global__ void __launch_bounds__(kThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tmx,
                        const __grid_constant__ CUtensorMap tmq,
                        const __grid_constant__ CUtensorMap tms, uint16_t* __restrict__ y, int M,
                        int N, int K, int tm, int mblocks, unsigned int* err) {
  extern __shared__ __align__(1024) char smem_raw[];
  char* sm = align1024(smem_raw);
  const uint32_t sb = smem_u32(sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cid = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
  auto bar = [&](int i) { return sb + kBarOff + 8u * (uint32_t)i; };
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(sm + kMiscOff);
  const int nblocks = (N + 2 * TN - 1) / (2 * TN);
  const int tiles = mblocks * nblocks;
  const int kblocks = K / BK;
  const int th = tm >> 1;  // rows held by each CTA
  const uint32_t xbytes = (uint32_t)th * BK * 2;
  const uint32_t stride = kWBytes + xbytes + kQBytes + kSBytes;
  const int ns = min(kMaxStages, kRingBytes / (int)stride);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(bar(kFull + s), 1);
      mbar_init(bar(kWReady + s), kDeqWarps + 1);  // even CTA's dequant warps + the relay
      mbar_init(bar(kPReady + s), kDeqWarps);      // odd CTA's dequant warps
      mbar_init(bar(kConsumed + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kAccFull + b), 1);
      mbar_init(bar(kAccEmpty + b), 2 * kEpiWarps);
    }
    mbar_init(bar(kDrain), 1);
    misc[1] = 0;
    mbar_fence_init();
  }
  if (warp == kMmaWarp) tc::tmem_alloc_pair(sb + kMiscOff, kTmemCols);
  tc::fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer's barriers are initialised before anyone arrives on them
  tc::fence_after();
  const uint32_t tmem = misc[0];

  auto fail = [&]() {
    if (err) atomicCAS(err, 0u, 8u);  // W4A16_ERR_TIMEOUT
    misc[1] = 1;
  };
  auto aborted = [&]() { return misc[1] != 0; };

  if (warp == kProdWarp) {
    if (lane == 0) {
      const uint32_t tx = xbytes + kQBytes + kSBytes;
      int it = 0;
      RingPos r;
      for (int tile = cid; tile < tiles && !aborted(); tile += nclusters) {
        const int mb = tile % mblocks, nb = tile / mblocks;
        const int col0 = nb * 2 * TN + (int)rank * TN, row0 = mb * tm + (int)rank * th;
        for (int kb = 0; kb < kblocks; ++kb, ++it, r.next(ns)) {
          if (!PF_WAIT(bar(kConsumed + r.s), r.ph ^ 1u, kWaitLimitNs) || aborted()) {
            fail();
            break;
          }
          const uint32_t st = sb + r.s * stride + kWBytes, full = bar(kFull + r.s);
          mbar_expect_tx(full, tx);
          tma_load_3d(st, &tmx, kb * BK, row0, 0, full);
          tma_load_3d(st + xbytes, &tmq, col0, kb * (BK / 8), 0, full);
          tma_load_3d(st + xbytes + kQBytes, &tms, col0, kb * (BK / 32), 0, full);
        }
      }
      // Let the last copies land before the CTA can exit (they target this CTA's memory).
      for (int j = (it > ns ? it - ns : 0); j < it; ++j)
        (void)mbar_wait(bar(kFull + j % ns), (j / ns) & 1, kWaitLimitNs / 16);
    }
  } else if (warp == kRelayWarp) {
    // Odd CTA: one thread waits for the local dequant barrier of each stage, releases the CTA's
    // shared-memory writes at cluster scope and arrives on the even CTA's wready. One thread per
    // CTA pays for the release instead of each of the 8 dequant warps.
    if (rank == 1 && lane == 0) {
      RingPos r;
      bool ok = true;
      for (int tile = cid; tile < tiles && ok && !aborted(); tile += nclusters) {
        for (int kb = 0; kb < kblocks; ++kb, r.next(ns)) {
          if (!PF_WAIT(bar(kPReady + r.s), r.ph, kWaitLimitNs) || aborted()) {
            fail();
            ok = false;
            break;
          }
          fence_release_shared_cluster();
          mbar_arrive_remote_relaxed(mapa_shared(bar(kWReady + r.s), 0));
        }
      }
    }
  } else if (warp >= kDeqWarp0) {
    // Thread = weight column n of this CTA's 128 and scale group h of the 64-deep k-block (words
    // 4h .. 4h + 3).
    const int n = ((warp - kDeqWarp0) % (TN / 32)) * 32 + lane;
    const int h = (warp - kDeqWarp0) / (TN / 32);
    const uint32_t wrow = (uint32_t)(n >> 3) * 1024u + (uint32_t)(n & 7) * 128u;
    RingPos r;
    for (int tile = cid; tile < tiles && !aborted(); tile += nclusters) {
      for (int kb = 0; kb < kblocks; ++kb, r.next(ns)) {
        if (!PF_WAIT(bar(kFull + r.s), r.ph, kWaitLimitNs) || aborted()) {
          fail();
          break;
        }
        const uint32_t st = sb + r.s * stride;
        const uint32_t q = st + kWBytes + xbytes + (4 * h * TN + n) * 4;
        const float sv = lds32f(st + kWBytes + xbytes + kQBytes + (h * TN + n) * 4);
        const __nv_bfloat162 hv = __floats2bfloat162_rn(sv, sv);
        const uint32_t s2 = *reinterpret_cast<const uint32_t*>(&hv);
        uint32_t w[4];
#pragma unroll
        for (int ii = 0; ii < 4; ++ii)
          asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(w[ii]) : "r"(q + ii * TN * 4));
#pragma unroll
        for (int ii = 0; ii < 4; ++ii) {
          const int i = 4 * h + ii;  // word (8 consecutive k) within the k-block
          const uint4 o = dequant_word_bf16(w[ii], s2);
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(
                           st + wrow + (uint32_t)((i ^ (n & 7)) << 4)),
                       "r"(o.x), "r"(o.y), "r"(o.z), "r"(o.w)
                       : "memory");
        }
        tc::fence_proxy_async();  // make the generic-proxy stores visible to the tensor cores
        __syncwarp();
        if (lane == 0) {
          tc::mbar_arrive(bar((rank == 0 ? kWReady : kPReady) + r.s));
        }
      }
    }
  } else if (warp == kMmaWarp) {
    if (rank == 0 && lane == 0) {
      const uint32_t idesc = kIdescNoN | ((uint32_t)(tm >> 3) << 17);
      const uint64_t adesc0 = tc::sw128_desc(sb);
      int tcount = 0;
      RingPos r;
      bool ok = true;
      for (int tile = cid; tile < tiles && ok && !aborted(); tile += nclusters, ++tcount) {
        const int b = tcount & 1, ause = tcount >> 1;
        if (!mbar_wait_cluster(bar(kAccEmpty + b), (ause & 1) ^ 1, kWaitLimitNs)) {
          fail();
          break;
        }
        tc::fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(b * kAccCols);
        for (int kb = 0; kb < kblocks; ++kb, r.next(ns)) {
          if (!mbar_wait_cluster(bar(kWReady + r.s), r.ph, kWaitLimitNs)) {
            fail();
            ok = false;
            break;
          }
          fence_acquire_shared_cluster();  // the odd CTA's weight tile and x half
          tc::fence_after();
          const uint64_t ad = adesc0 + (uint64_t)((r.s * stride) >> 4);
          const uint64_t bd = ad + (kWBytes >> 4);
          tc::mma_ss_pair(d_tmem, ad, bd, idesc, kb > 0 ? 1u : 0u);
#pragma unroll
          for (int kk = 1; kk < BK / 16; ++kk)
            tc::mma_ss_pair(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc, 1u);
          tc::commit_pair(bar(kConsumed + r.s), (uint16_t)3);  // frees the stage in both CTAs
        }
        if (!ok) break;
        tc::commit_pair(bar(kAccFull + b), (uint16_t)3);  // accumulator complete in both
      }
      // All MMAs issued by this thread have finished before either CTA releases TMEM.
      tc::commit_pair(bar(kDrain), (uint16_t)1);
      (void)mbar_wait(bar(kDrain), 0, kWaitLimitNs);
    }
  } else {  // epilogue warps 0..3: TMEM lanes 32*warp .. 32*warp + 31 = weight columns
    int tcount = 0;
    for (int tile = cid; tile < tiles && !aborted(); tile += nclusters, ++tcount) {
      const int mb = tile % mblocks, nb = tile / mblocks;
      const int b = tcount & 1, ause = tcount >> 1;
      if (!mbar_wait_cluster(bar(kAccFull + b), ause & 1, kWaitLimitNs)) {
        fail();
        break;
      }
      tc::fence_after();
      const int n = nb * 2 * TN + (int)rank * TN + warp * 32 + lane;
      const int rows = min(tm, M - mb * tm);
      uint16_t* yc = y + (size_t)mb * tm * N + n;
      const uint32_t tbase = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(b * kAccCols);
#pragma unroll 1
      for (int cc = 0; cc < (rows + 31) / 32; ++cc) {
        uint32_t rr[32];
        tc::tmem_ld32(tbase + cc * 32, rr);
        tc::tmem_wait_ld(rr);
        if (n < N) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (cc * 32 + j < rows)
              yc[(size_t)(cc * 32 + j) * N] = __bfloat16_as_ushort(
                  __float2bfloat16_rn(__uint_as_float(rr[j])));
          }
        }
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(bar(kAccEmpty + b), 0));
    }
  }

  tc::fence_before();
  __syncthreads();
  cluster_sync_all();  // neither CTA leaves while the pair's MMAs or arrivals may touch it
  tc::fence_after();
  if (warp == kMmaWarp) tc::tmem_dealloc_pair(tmem, kTmemCols);
}

}  // namespace

// Row blocks of at most 256 rows, split evenly: tm = M / ceil(M / 256) rounded up to 16. One
// cluster of two CTAs per pair of SMs (as many as can be resident), persistent over the tiles.
cudaError_t launch_gemm_bf16(const uint16_t* x, const int32_t* qw, const float* sc, uint16_t* y,
                             int M, int N, int K, cudaStream_t s) {
  DeviceInfo di;
  cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return e;
  static PerDeviceOnce<int> pairs_cache;  // resident CTA pairs
  const int* max_pairs = nullptr;
  e = pairs_cache.get(di.device, [&](int& pairs) {
    cudaError_t r = cudaFuncSetAttribute(prefill_pair_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (r != cudaSuccess) return r;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = kSmemAlloc;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int nc = 0;
    if (cudaOccupancyMaxActiveClusters(&nc, prefill_pair_kernel, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      nc = 0;
    }
    pairs = nc > 0 ? nc : di.sm_count / 2;
    return cudaSuccess;
  }, &max_pairs);
  if (e != cudaSuccess) return e;
  const int mblocks = (M + TM - 1) / TM;
  const int tm = (((M + mblocks - 1) / mblocks) + 15) / 16 * 16;
  CUtensorMap tmx, tmq, tms;
  e = make_tmap_ex(&tmx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, CU_TENSOR_MAP_SWIZZLE_128B, x,
                   (uint64_t)K, (uint64_t)M, 1, BK, tm / 2);
  if (e != cudaSuccess) return e;
  e = make_tmap_ex(&tmq, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, CU_TENSOR_MAP_SWIZZLE_NONE, qw,
                   (uint64_t)N, (uint64_t)(K / 8), 1, TN, BK / 8);
  if (e != cudaSuccess) return e;
  e = make_tmap_ex(&tms, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, CU_TENSOR_MAP_SWIZZLE_NONE, sc,
                   (uint64_t)N, (uint64_t)(K / kGroup), 1, TN, BK / 32);
  if (e != cudaSuccess) return e;
  const int tiles = mblocks * ((N + 2 * TN - 1) / (2 * TN));
  const int pairs = tiles < *max_pairs ? tiles : *max_pairs;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemAlloc;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_pair_kernel, tmx, tmq, tms, y, M, N, K, tm, mblocks,
                            device_error_word());
}

}  // namespace w4a16
