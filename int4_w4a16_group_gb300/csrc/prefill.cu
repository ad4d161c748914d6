// Large-M (prefill) contraction on the 5th-generation tensor cores (tcgen05, TMEM, TMA):
//   y[M, N] (bf16) = x[M, K] (bf16) @ bf16(dequant(qw, sc)) with float32 accumulation.
// The pages' activations are float32 and their kernel has no large-M form; this path serves
// batched prefill, where the op really is a dense contraction.
//
// Persistent CTAs (one per SM) walk 128 x BN output tiles (BN = 256, or 128 when the wide tiles
// would leave SMs idle), M-blocks fastest so the x tiles of a weight block are reused from L2.
// Per 64-deep K block of a tile:
//   * a TMA producer warp loads the x tile (128 x 64 bf16, 128-byte swizzle = the UMMA K-major
//     canonical layout), 8 packed rows x BN columns of codes and 2 rows of scales into a 5-stage
//     ring;
//   * dequant warps (two threads per weight column, one per group of the k-block) turn each
//     packed word (8 consecutive k of one column) into 8 bf16 values:
//     ((w >> 4j) & 0x000F000F) | 0x43004300 is the bf16 pair (128 + n_j, 128 + n_{j+4}); a bf16
//     FMA subtracts 136 exactly, another multiplies by the bf16 group scale; byte permutes
//     restore k order; one 16-byte store puts them in the swizzled K-major B tile of a separate
//     2-stage ring;
//   * one thread issues 4 tcgen05.mma (M = 128, N = BN, K = 16, bf16 x bf16 -> f32) into a TMEM
//     accumulator and commits to the barriers that free the x/codes stage and the B tile;
//   * 4 epilogue warps drain the finished accumulator (double-buffered, 2 x BN TMEM columns)
//     with tcgen05.ld, round to bf16 and store.
// Every barrier wait is bounded; a timeout sets the device error word and the CTA winds down.
#include <cuda_bf16.h>

#include "internal.h"
#include "mma_core.cuh"
#include "tc_core.cuh"

namespace w4a16 {
namespace {

using namespace mma;

constexpr int BM = 128, BK = 64;
// Two rings: the TMA ring of x tiles, codes and scales (kStagesA), and the ring of dequantized
// bf16 B tiles (kStagesB), so TMA can run further ahead than the dequant warps need B tiles.
#ifndef W4A16_PREFILL_STAGES_A
#define W4A16_PREFILL_STAGES_A 5
#endif
#ifndef W4A16_PREFILL_STAGES_B
#define W4A16_PREFILL_STAGES_B 2
#endif
constexpr int kStagesA = W4A16_PREFILL_STAGES_A;
constexpr int kStagesB = W4A16_PREFILL_STAGES_B;
constexpr int kEpiWarps = 4;  // warps 0..3 (TMEM lane quadrants 0..3)
constexpr int kProdWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kDeqWarp0 = 6;
#ifndef W4A16_PREFILL_DEQ_SPLIT
#define W4A16_PREFILL_DEQ_SPLIT 2
#endif
// threads per weight column (each takes one group of the 64-deep k-block when 2)
constexpr int kDeqSplit = W4A16_PREFILL_DEQ_SPLIT;
static_assert(kDeqSplit == 1 || kDeqSplit == 2, "a 64-deep k-block holds two groups");
// Everything that depends on the tile width BN (weight columns per tile: 256, or 128 when 256-wide
// tiles would leave SMs idle).
template <int BN_>
struct PF {
  static constexpr int BN = BN_;
  static constexpr int kDeqWarps = kDeqSplit * BN / 32;
  static constexpr int kThreads = (kDeqWarp0 + kDeqWarps) * 32;
  static constexpr int kAccCols = BN;
  static constexpr int kTmemCols = 2 * kAccCols;
  static constexpr int kABytes = BM * BK * 2;
  static constexpr int kBBytes = BN * BK * 2;
  static constexpr int kQBytes = (BK / 8) * BN * 4;
  static constexpr int kSBytes = (BK / 32) * BN * 4;
  static constexpr int kAOff = 0;
  static constexpr int kQOff = kAOff + kStagesA * kABytes;
  static constexpr int kSOff = kQOff + kStagesA * kQBytes;
  static constexpr int kBOff = ((kSOff + kStagesA * kSBytes + 1023) / 1024) * 1024;  // SW128 tiles
  static constexpr int kBarOff = kBOff + kStagesB * kBBytes;
  // barriers: full[SA] | empty[SA] | bready[SB] | bempty[SB] | accfull[2] | accempty[2] | drain
  static constexpr int kFull = 0, kEmpty = kStagesA, kBReady = 2 * kStagesA,
                       kBEmpty = 2 * kStagesA + kStagesB, kAccFull = 2 * kStagesA + 2 * kStagesB,
                       kAccEmpty = kAccFull + 2, kDrain = kAccEmpty + 2;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // [0] TMEM base, [1] abort flag
  static constexpr int kSmemBytes = kMiscOff + 16;
  static constexpr int kSmemAlloc = kSmemBytes + 1024;
  static constexpr uint32_t kStageTx = kABytes + kQBytes + kSBytes;
  // Instruction descriptor: bf16 x bf16 -> f32, M = 128, N = BN, both operands K-major.
  static constexpr uint32_t kIdesc = tc::idesc_f16(true, BM, BN);
  static_assert(kSmemAlloc <= 227 * 1024, "shared memory per CTA");
};

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

template <int BN>
__global__ void __launch_bounds__(PF<BN>::kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmq,
                   const __grid_constant__ CUtensorMap tms, uint16_t* __restrict__ y, int M,
                   int N, int K, unsigned int* err) {
  using C = PF<BN>;
  extern __shared__ __align__(1024) char smem_raw[];
  char* sm = align1024(smem_raw);
  const uint32_t sb = smem_u32(sm);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto bar = [&](int i) { return sb + C::kBarOff + 8u * (uint32_t)i; };
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(sm + C::kMiscOff);
  const int mblocks = (M + BM - 1) / BM, nblocks = (N + BN - 1) / BN;
  const int tiles = mblocks * nblocks;
  const int kblocks = K / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesA; ++s) {
      mbar_init(bar(C::kFull + s), 1);
      mbar_init(bar(C::kEmpty + s), 1);
    }
    for (int s = 0; s < kStagesB; ++s) {
      mbar_init(bar(C::kBReady + s), C::kDeqWarps);
      mbar_init(bar(C::kBEmpty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(C::kAccFull + b), 1);
      mbar_init(bar(C::kAccEmpty + b), kEpiWarps);
    }
    mbar_init(bar(C::kDrain), 1);
    misc[1] = 0;
    mbar_fence_init();
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(sb + C::kMiscOff, C::kTmemCols);
  }
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tmem = misc[0];

  auto fail = [&]() {
    if (err) atomicCAS(err, 0u, 8u);  // W4A16_ERR_TIMEOUT
    misc[1] = 1;
  };
  auto aborted = [&]() { return misc[1] != 0; };

  if (warp == kProdWarp) {
    if (lane == 0) {
      int it = 0;
      for (int tile = blockIdx.x; tile < tiles && !aborted(); tile += gridDim.x) {
        const int mb = tile % mblocks, nb = tile / mblocks;
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int s = it % kStagesA, use = it / kStagesA;
          if (!mbar_wait(bar(C::kEmpty + s), (use & 1) ^ 1, kWaitLimitNs) || aborted()) {
            fail();
            break;
          }
          mbar_expect_tx(bar(C::kFull + s), C::kStageTx);
          tma_load_3d(sb + C::kAOff + s * C::kABytes, &tmx, kb * BK, mb * BM, 0, bar(C::kFull + s));
          tma_load_3d(sb + C::kQOff + s * C::kQBytes, &tmq, nb * BN, kb * (BK / 8), 0,
                      bar(C::kFull + s));
          tma_load_3d(sb + C::kSOff + s * C::kSBytes, &tms, nb * BN, kb * (BK / 32), 0,
                      bar(C::kFull + s));
        }
      }
      // Let the last copies land before the CTA can exit (they target this CTA's memory).
      for (int j = (it > kStagesA ? it - kStagesA : 0); j < it; ++j)
        (void)mbar_wait(bar(C::kFull + j % kStagesA), (j / kStagesA) & 1, kWaitLimitNs / 16);
    }
  } else if (warp >= kDeqWarp0) {
    // Thread = weight column n of the tile and, with two threads per column, group h of the
    // 64-deep k-block (words 4h .. 4h + 3).
    constexpr int kWords = (BK / 8) / kDeqSplit;
    const int n = ((warp - kDeqWarp0) % (BN / 32)) * 32 + lane;
    const int h = (warp - kDeqWarp0) / (BN / 32);
    const uint32_t brow = (uint32_t)(n >> 3) * 1024u + (uint32_t)(n & 7) * 128u;
    int it = 0;
    for (int tile = blockIdx.x; tile < tiles && !aborted(); tile += gridDim.x) {
      for (int kb = 0; kb < kblocks; ++kb, ++it) {
        const int s = it % kStagesA, use = it / kStagesA;
        const int sbt = it % kStagesB, useb = it / kStagesB;
        if (!mbar_wait(bar(C::kFull + s), use & 1, kWaitLimitNs) ||
            !mbar_wait(bar(C::kBEmpty + sbt), (useb & 1) ^ 1, kWaitLimitNs) || aborted()) {
          fail();
          break;
        }
        const uint32_t q = sb + C::kQOff + s * C::kQBytes + (h * kWords * BN + n) * 4;
        const uint32_t sc = sb + C::kSOff + s * C::kSBytes + n * 4;
        // bf16 scale pair of each group this thread covers (group g of the k-block = words
        // 4g .. 4g + 3).
        uint32_t s2[2];
#pragma unroll
        for (int gq = 0; gq < 2 / kDeqSplit; ++gq) {
          const float sv = lds32f(sc + (h * (2 / kDeqSplit) + gq) * BN * 4);
          const __nv_bfloat162 hv = __floats2bfloat162_rn(sv, sv);
          s2[gq] = *reinterpret_cast<const uint32_t*>(&hv);
        }
        const uint32_t bbase = sb + C::kBOff + sbt * C::kBBytes + brow;
#pragma unroll
        for (int ii = 0; ii < kWords; ++ii) {
          const int i = h * kWords + ii;  // word (8 consecutive k) within the k-block
          uint32_t w;
          asm volatile("ld.shared.b32 %0, [%1];\n" : "=r"(w) : "r"(q + ii * BN * 4));
          const uint4 o = dequant_word_bf16(w, s2[ii >> 2]);
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(
                           bbase + (uint32_t)((i ^ (n & 7)) << 4)),
                       "r"(o.x), "r"(o.y), "r"(o.z), "r"(o.w)
                       : "memory");
        }
        tc::fence_proxy_async();  // make the generic-proxy stores visible to the tensor cores
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(bar(C::kBReady + sbt));
      }
    }
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      int it = 0, tcount = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < tiles && ok && !aborted(); tile += gridDim.x, ++tcount) {
        const int b = tcount & 1, ause = tcount >> 1;
        if (!mbar_wait(bar(C::kAccEmpty + b), (ause & 1) ^ 1, kWaitLimitNs)) {
          fail();
          break;
        }
        tc::fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(b * C::kAccCols);
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int s = it % kStagesA, use = it / kStagesA;
          const int sbt = it % kStagesB, useb = it / kStagesB;
          if (!mbar_wait(bar(C::kFull + s), use & 1, kWaitLimitNs) ||
              !mbar_wait(bar(C::kBReady + sbt), useb & 1, kWaitLimitNs) || aborted()) {
            fail();
            ok = false;
            break;
          }
          tc::fence_after();
          const uint32_t a0 = sb + C::kAOff + s * C::kABytes, b0 = sb + C::kBOff + sbt * C::kBBytes;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc::mma_ss(d_tmem, tc::sw128_desc(a0 + kk * 32), tc::sw128_desc(b0 + kk * 32),
                       C::kIdesc, (kb > 0 || kk > 0) ? 1u : 0u);
          tc::commit(bar(C::kEmpty + s));     // frees the x/codes stage once these MMAs read it
          tc::commit(bar(C::kBEmpty + sbt));  // and the B tile
        }
        if (!ok) break;
        tc::commit(bar(C::kAccFull + b));  // accumulator complete
      }
      // All MMAs issued by this thread have finished before TMEM is released.
      tc::commit(bar(C::kDrain));
      (void)mbar_wait(bar(C::kDrain), 0, kWaitLimitNs);
    }
  } else {  // epilogue warps 0..3: TMEM lanes 32*warp .. 32*warp + 31 = tile rows
    int tcount = 0;
    for (int tile = blockIdx.x; tile < tiles && !aborted(); tile += gridDim.x, ++tcount) {
      const int mb = tile % mblocks, nb = tile / mblocks;
      const int b = tcount & 1, ause = tcount >> 1;
      if (!mbar_wait(bar(C::kAccFull + b), ause & 1, kWaitLimitNs)) {
        fail();
        break;
      }
      tc::fence_after();
      const int row = mb * BM + warp * 32 + lane;
      const uint32_t tbase = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(b * C::kAccCols);
#pragma unroll 1
      for (int cc = 0; cc < BN / 32; ++cc) {
        uint32_t r[32];
        tc::tmem_ld32(tbase + cc * 32, r);
        tc::tmem_wait_ld(r);
        if (row < M) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int col = nb * BN + cc * 32 + 8 * j;
            if (col < N) {
              uint32_t o[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 hv = __floats2bfloat162_rn(
                    __uint_as_float(r[8 * j + 2 * e]), __uint_as_float(r[8 * j + 2 * e + 1]));
                o[e] = *reinterpret_cast<const uint32_t*>(&hv);
              }
              *reinterpret_cast<uint4*>(y + (size_t)row * N + col) =
                  make_uint4(o[0], o[1], o[2], o[3]);
            }
          }
        }
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(bar(C::kAccEmpty + b));
    }
  }

  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == kMmaWarp) tc::tmem_dealloc(tmem, C::kTmemCols);
}

template <int BN>
cudaError_t launch_prefill(const uint16_t* x, const int32_t* qw, const float* sc, uint16_t* y,
                           int M, int N, int K, const DeviceInfo& di, cudaStream_t s) {
  using C = PF<BN>;
  static int attr_devices = 0;
  const int bit = 1 << (di.device & 31);
  if (!(attr_devices & bit)) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<BN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemAlloc);
    if (e != cudaSuccess) return e;
    attr_devices |= bit;
  }
  CUtensorMap tmx, tmq, tms;
  cudaError_t e = make_tmap_ex(&tmx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                               CU_TENSOR_MAP_SWIZZLE_128B, x, (uint64_t)K, (uint64_t)M, 1, BK, BM);
  if (e != cudaSuccess) return e;
  e = make_tmap_ex(&tmq, CU_TENSOR_MAP_DATA_TYPE_INT32, 4, CU_TENSOR_MAP_SWIZZLE_NONE, qw,
                   (uint64_t)N, (uint64_t)(K / 8), 1, BN, BK / 8);
  if (e != cudaSuccess) return e;
  e = make_tmap_ex(&tms, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, CU_TENSOR_MAP_SWIZZLE_NONE, sc,
                   (uint64_t)N, (uint64_t)(K / kGroup), 1, BN, BK / 32);
  if (e != cudaSuccess) return e;
  const int tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  const int grid = tiles < di.sm_count ? tiles : di.sm_count;
  prefill_kernel<BN><<<grid, C::kThreads, C::kSmemAlloc, s>>>(tmx, tmq, tms, y, M, N, K,
                                                                device_error_word());
  return cudaGetLastError();
}

}  // namespace

// 128 x 256 tiles by default; 128 x 128 tiles when even twice as many tiles fit in one wave over
// the SMs (then the wide tiles would leave more than half of them idle).
cudaError_t launch_gemm_bf16(const uint16_t* x, const int32_t* qw, const float* sc, uint16_t* y,
                             int M, int N, int K, cudaStream_t s) {
  DeviceInfo di;
  cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return e;
  const long long wide_tiles = (long long)((M + BM - 1) / BM) * ((N + 255) / 256);
  return 2 * wide_tiles <= di.sm_count ? launch_prefill<128>(x, qw, sc, y, M, N, K, di, s)
                                       : launch_prefill<256>(x, qw, sc, y, M, N, K, di, s);
}

}  // namespace w4a16
