// Warp-specialized weight-streaming core for small M (decode / draft-tree verify rows).
//
// Page "The Weight of Precision: Building Native INT4 Quantization for a Custom Speculative
// Decoding Engine", section "The Kernel: w4a16_gemm": y = x @ dequant(W) with FP32 activations,
// INT4 codes (nibble - 8, eight per int32 along K) and one float32 scale per 32 input rows per
// output column. The pages measure the optimized kernel against HBM bandwidth, so every packed
// weight and scale byte is streamed exactly once and the per-weight instruction count is what
// this core minimizes.
//
// A CTA has three roles:
//   * producer warp (one elected lane): per stage of G groups (4G packed rows) one TMA copy of
//     the codes of all the CTA's 32-column tiles (a 4-D/5-D box: columns x rows x tiles
//     [x gate/up half] x matrix, the last coordinate picking an expert of stacked MoE weights)
//     and one of their scales, into an R-stage ring (full/empty mbarriers);
//   * prep warp: TMA-loads raw activation chunks (CG groups x up to 16 rows), finds each row's
//     largest magnitude in the chunk, and writes the rows as MMA B-fragments in fp16: the row
//     scaled by 2^(14 - e) (e = the row's exponent in this chunk) split into hi + lo terms, 22
//     significant bits of each float32 value (bf16 activations need only the hi term, exactly);
//   * W consumer warps: per group, per 32-column tile: one 16-byte shared load of codes, one of
//     scales, the fp16 magic-number unpack (nibble | 0x6400 is 1024 + nibble; one fp16 FMA
//     gives nibble - 8 exactly), mma.sync m16n8k16 (fp16 x fp16 -> fp32), and one FMA per output
//     applying the group scale. The chunk exponents are applied to the accumulators only when a
//     chunk ends (a power-of-two rescale), so there is no per-group multiply.
// Products of exact codes and fp16 terms are exact in fp32; the only rounding beyond float32
// accumulation is the 2^-22 relative cut of each activation.
//
// Orientation (m16n8k16, g = lane / 4, t = lane % 4): A = 16 weight columns x 16 k (the codes),
// B = 16 k x 8 activation columns, C = 16 x 8. Lane (g, t) reads the 16-byte chunk
// h(g) = g/2 + 4 (g%2) of packed row 4j + t (columns 4h .. 4h + 3) of each tile; A tile T uses
// columns 4h + 2T (A row g) and 4h + 2T + 1 (A row g + 8). The k order inside a group is
// permuted identically in A and B (k-slot 2t + {0,1} = input 8t + {0,4}, 2t + 8 + {0,1} =
// 8t + {1,5} in the first k-step; 8t + {2,6}, 8t + {3,7} in the second), which the sum ignores.
// B columns by mode:
//   kN2 (up to 4 rows):  B column n = (row n/2, term n%2): both terms in one MMA column pair.
//   kK2 (8 rows/block):  B column n = row 8b + n; hi and lo terms are two k-passes over the same
//                        A fragments, summed by the MMA itself.
//   kK1 (8 rows/block):  one term (bf16 activations are exact in fp16 after the exponent shift).
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mma_core.cuh"

namespace w4a16 {
namespace ws {

using mma::lds128;
using mma::mbar_expect_tx;
using mma::mbar_init;
using mma::mbar_try_wait;
using mma::smem_u32;

enum Mode { kN2 = 0, kK2 = 1, kK1 = 2 };

using mma::kWaitLimitNs;

// ------------------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, int c3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, int c3, int c4, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
      "r"(bar)
      : "memory");
}
// Plain arrive (release at CTA scope) on a barrier of this CTA.
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
// Orders this thread's earlier generic-proxy accesses of shared memory before later async-proxy
// (TMA) accesses of it.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];\n" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Programmatic dependent launch: a grid launched with programmatic stream serialization may
// start before the previous kernel on its stream has finished. dependency_wait() blocks the
// calling thread until that kernel has completed and its memory is visible (a no-op when the
// grid was launched normally); allow_dependents() lets the next such grid be scheduled.
__device__ __forceinline__ void dependency_wait() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
}
__device__ __forceinline__ void allow_dependents() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// Bounded wait on phase `parity`: sleeps in steps of at most 1 ms; gives up (false) when the
// CTA's abort flag is raised or after kWaitLimitNs.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity,
                                           const volatile int* abort_flag) {
  constexpr uint32_t kStepNs = 1000000u;
  if (mbar_try_wait(bar, parity, kStepNs)) return true;
  const uint64_t t0 = mma::global_ns();
  while (!mbar_try_wait(bar, parity, kStepNs)) {
    if (*abort_flag || mma::global_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// As wait_phase, but polls: try_wait without a sleep hint (the hardware's own short suspend), for
// the consumer warps, whose wake-up latency is on the critical path.
__device__ __forceinline__ bool wait_phase_poll(uint32_t bar, uint32_t parity,
                                                const volatile int* abort_flag) {
  if (mma::mbar_try_wait_poll(bar, parity)) return true;
  const uint64_t t0 = mma::global_ns();
  uint32_t n = 0;
  while (!mma::mbar_try_wait_poll(bar, parity)) {
    if ((++n & 255u) == 0 && (*abort_flag || mma::global_ns() - t0 > kWaitLimitNs)) return false;
  }
  return true;
}
#ifndef W4A16_POLL_CONSUMER
#define W4A16_POLL_CONSUMER 0
#endif
__device__ __forceinline__ bool wait_consumer(uint32_t bar, uint32_t parity,
                                              const volatile int* abort_flag) {
  return W4A16_POLL_CONSUMER ? wait_phase_poll(bar, parity, abort_flag)
                             : wait_phase(bar, parity, abort_flag);
}

// Records a wait that gave up: the library's error word (W4A16_ERR_TIMEOUT) and the CTA's abort
// flag, so the other roles stop waiting for work that will not come.
__device__ __forceinline__ void raise_abort(volatile int* abort_flag, unsigned int* err) {
  *abort_flag = 1;
  if (err) atomicCAS(err, 0u, 8u);
}

// ------------------------------------------------------------------------------ geometry

// Rows of activations one CTA serves, by mode and MMA column blocks.
template <int MODE, int NB>
struct ModeInfo {
  static_assert(MODE != kN2 || NB == 1, "the two-term-column mode has one block of 4 rows");
  static constexpr int kRowsPerBlock = MODE == kN2 ? 4 : 8;
  static constexpr int kRows = kRowsPerBlock * NB;
  static constexpr int kTerms = MODE == kK1 ? 1 : 2;
  // B-fragment bytes per group: 512 per (block, term) chunk (32 lanes x 16 B); kN2 holds both
  // terms in one chunk.
  static constexpr int kFragGroup = MODE == kN2 ? 512 : NB * kTerms * 512;
};

// Shared-memory layout of one CTA (offsets from a 1024-byte aligned base):
//   codes  R stages x kTiles x (4G x 128 B, 128-byte swizzle)
//   scales R stages x kTiles x (G x 128 B)
//   xraw   2 x (kRows x 32 CG activations)         -- raw activation chunks (TMA)
//   frag   2 x (CG x kFragGroup)                   -- prepared B fragments
//   fexp   2 x kExpInts ints                       -- row exponents (up to 32) and a changed flag
//   bars   full[R], empty[R], xfull[2], ffull[2], fempty[2]; abort flag
// CG = groups per activation chunk (at most 8: a TMA box row holds at most 256 elements).
template <int MODE, int NB, int W, int CH, int G, int R, int CG, int XBYTES>
struct WsGeo {
  using MI = ModeInfo<MODE, NB>;
  static constexpr int kMode = MODE;
  static constexpr int kNB = NB;
  static constexpr int kW = W;
  static constexpr int kCH = CH;
  static constexpr int kG = G;
  static constexpr int kR = R;
  static constexpr int kCG = CG;
  static constexpr int kConsumers = W;
  static constexpr int kThreads = 32 * (W + 2);
  static constexpr int kTiles = W * CH;
  static constexpr int kCodeTile = 4 * G * 128;
  static constexpr int kScaleTile = G * 128;
  static constexpr int kCodeStage = kTiles * kCodeTile;
  static constexpr int kScaleStage = kTiles * kScaleTile;
  static constexpr uint32_t kStageTx = kCodeStage + kScaleStage;
  static constexpr int kXRawBytes = MI::kRows * CG * 32 * XBYTES;
  static constexpr int kFragBytes = CG * MI::kFragGroup;
  static constexpr int kCodeOff = 0;
  static constexpr int kScaleOff = kCodeOff + R * kCodeStage;
  static constexpr int kXRawOff = kScaleOff + R * kScaleStage;
  static constexpr int kFragOff = kXRawOff + 2 * kXRawBytes;
  static constexpr int kExpOff = kFragOff + 2 * kFragBytes;
  static constexpr int kExpInts = 64;  // per buffer: row exponents [0, 32), changed flag at 32
  static constexpr int kExpFlag = 32;
  static constexpr int kBarOff = kExpOff + 2 * kExpInts * 4;
  static constexpr int kNumBars = 2 * R + 7;  // + the split-K receive barrier
  static constexpr int kAbortOff = kBarOff + kNumBars * 8;
  static constexpr int kBytes = kAbortOff + 16;
  static constexpr int kAlloc = kBytes + 1024;  // room to align the base
  static_assert(G % 2 == 0, "a tile's rows must fill whole 1 KB swizzle periods");
  static_assert(MI::kRows <= kExpFlag, "row exponents must fit below the changed flag");
  static_assert(CG % G == 0 && CG <= 8, "a chunk is a whole number of stages, <= 256 inputs");
  static_assert((kCodeStage % 1024) == 0 && (kScaleOff % 1024) == 0, "TMA destinations");
  static_assert((kXRawOff % 128) == 0 && (kFragOff % 128) == 0, "16-byte aligned buffers");
};

// ------------------------------------------------------------------------------ prep warp

// Exponent of a row's largest magnitude (|x| < 2^(e+1)); kNoExp for an all-zero row. Every
// finite float32 has e <= 127, so scaled by 2^(14 - e) it stays below 2^15. The lower clamp
// keeps 2^(14 - e), the output factor 2^(e - 14) and the rescale factors between chunks
// (two halves of 2^(e_old - e_new)) normal floats; rows whose largest magnitude is below
// 2^-100 are scaled as if it were 2^-100 and keep fewer significant bits.
constexpr int kNoExp = -1000;
__device__ __forceinline__ int row_exponent(float amax) {
  if (amax == 0.0f) return kNoExp;
  const int ex = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127;
  return ex < -100 ? -100 : ex;
}

__device__ __forceinline__ float load_act(const float* p) { return *p; }

// Eight consecutive activations of a raw chunk row (16-byte aligned) as floats.
__device__ __forceinline__ void load8(uint32_t addr, const float*, float (&v)[8]) {
  const uint4 a = lds128(addr), b = lds128(addr + 16);
  v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y);
  v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
  v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y);
  v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
}
__device__ __forceinline__ void load8(uint32_t addr, const uint16_t*, float (&v)[8]) {
  const uint4 a = lds128(addr);  // 8 bf16 values: a bf16 is the top half of its float32
  v[0] = __uint_as_float(a.x << 16); v[1] = __uint_as_float(a.x & 0xFFFF0000u);
  v[2] = __uint_as_float(a.y << 16); v[3] = __uint_as_float(a.y & 0xFFFF0000u);
  v[4] = __uint_as_float(a.z << 16); v[5] = __uint_as_float(a.z & 0xFFFF0000u);
  v[6] = __uint_as_float(a.w << 16); v[7] = __uint_as_float(a.w & 0xFFFF0000u);
}

__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
  const __half2 p = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&p);
}

// Eight scaled activations -> the 16-byte B fragment of one term, in the codes' k order:
// (v0, v4), (v1, v5), (v2, v6), (v3, v7).
__device__ __forceinline__ uint4 frag_of(const float (&o)[8]) {
  return make_uint4(pack_h2(o[0], o[4]), pack_h2(o[1], o[5]), pack_h2(o[2], o[6]),
                    pack_h2(o[3], o[7]));
}

// Converts raw chunk `buf` (ngr groups) into B fragments and row exponents. Lane (g, t) of the
// prep warp writes exactly the 16-byte pieces consumer lane (g, t) will read.
// Row exponents are sticky downwards: a row keeps the exponent e of earlier chunks (eprev)
// while this chunk's largest magnitude is below 2^(e + 1), and takes the chunk's exponent when
// it is larger. Scaled by 2^(14 - e) every value is then below 2^15, well inside fp16 (whose
// largest finite value is 65504; round-to-nearest overflows from 65520, so a chunk one binade
// up could not be kept). The chunk's flag word tells the consumers whether any row's exponent
// changed (only then do they rescale their accumulators). `first` starts a new sequence.
template <int MODE, int NB, typename XT, typename L>
__device__ __forceinline__ void prep_chunk(char* base, int buf, int ngr,
                                           int (&eprev)[MODE == kN2 ? 1 : NB], bool first) {
  using MI = typename L::MI;
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  constexpr int kRowBytes = L::kCG * 32 * (int)sizeof(XT);
  const uint32_t raw = smem_u32(base + L::kXRawOff + buf * L::kXRawBytes);
  char* frag = base + L::kFragOff + buf * L::kFragBytes;
  int* fexp = reinterpret_cast<int*>(base + L::kExpOff) + buf * L::kExpInts;
  constexpr int kLaneRows = MODE == kN2 ? 1 : NB;  // rows this lane converts
  int rows[kLaneRows];
#pragma unroll
  for (int i = 0; i < kLaneRows; ++i) rows[i] = MODE == kN2 ? (g >> 1) : 8 * i + g;

  // Each row's largest magnitude over the chunk: lanes (g, t = 0..3) [and g ^ 1 for kN2] share
  // a row and see all of its inputs between them.
  int ex[kLaneRows];
#pragma unroll
  for (int i = 0; i < kLaneRows; ++i) {
    float amax = 0.0f;
    for (int j = 0; j < ngr; ++j) {
      float v[8];
      load8(raw + rows[i] * kRowBytes + (32 * j + 8 * t) * (int)sizeof(XT), (const XT*)nullptr, v);
#pragma unroll
      for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(v[e]));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const int ec = row_exponent(amax);
    // a row with no nonzero value so far takes the chunk's exponent
    ex[i] = (first || eprev[i] == kNoExp || ec > eprev[i]) ? ec : eprev[i];
    if (t == 0 && (MODE != kN2 || (g & 1) == 0)) fexp[rows[i]] = ex[i] == kNoExp ? 0 : ex[i];
  }
  bool changed = false;
#pragma unroll
  for (int i = 0; i < kLaneRows; ++i) {
    changed |= !first && ex[i] != eprev[i];
    eprev[i] = ex[i];
    if (ex[i] == kNoExp) ex[i] = 0;  // zero rows: any scale
  }
  changed = __any_sync(0xffffffffu, changed);
  if (lane == 0) fexp[L::kExpFlag] = changed ? 1 : 0;

  for (int j = 0; j < ngr; ++j) {
#pragma unroll
    for (int i = 0; i < kLaneRows; ++i) {
      float v[8];
      load8(raw + rows[i] * kRowBytes + (32 * j + 8 * t) * (int)sizeof(XT), (const XT*)nullptr, v);
      const float up = mma::exp2i(14 - ex[i]);
      float hi[8], lo[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float xs = v[e] * up;
        hi[e] = __half2float(__float2half_rn(xs));
        lo[e] = xs - hi[e];
      }
      char* dst = frag + j * MI::kFragGroup + lane * 16;
      if constexpr (MODE == kN2) {
        *reinterpret_cast<uint4*>(dst) = frag_of((g & 1) ? lo : hi);
      } else if constexpr (MODE == kK2) {
        *reinterpret_cast<uint4*>(dst + (2 * i) * 512) = frag_of(hi);
        *reinterpret_cast<uint4*>(dst + (2 * i + 1) * 512) = frag_of(lo);
      } else {
        *reinterpret_cast<uint4*>(dst + i * 512) = frag_of(hi);
      }
    }
  }
}

// ------------------------------------------------------------------------------ consumers

// Accumulators of one consumer lane: [tile c][A tile T][block b][C register r].
template <int CH, int NB>
struct Acc {
  float v[CH][2][NB][4];
};

// Shared-memory slot (within a stage) of tile c of consumer warp w. Plain: w*CH + c. Fused
// SwiGLU: gate tiles fill slots [0, kTiles/2) and the matching up tiles [kTiles/2, kTiles); a
// warp's tiles c < CH/2 are gate tiles, c >= CH/2 the matching up tiles.
template <int W, int CH, bool SWIGLU>
__device__ __forceinline__ int tile_slot(int w, int c) {
  static_assert(!SWIGLU || CH % 2 == 0, "a fused SwiGLU warp holds gate/up tile pairs");
  if constexpr (SWIGLU) {
    constexpr int H = CH / 2, TT = W * CH / 2;
    return c < H ? w * H + c : TT + w * H + (c - H);
  } else {
    return w * CH + c;
  }
}

// One group (32 inputs) of all CH tiles of this warp. code_j / scale_j address the group's
// packed rows and scale row in stage memory (lane offsets included); fr the group's fragments.
template <int MODE, int NB, int W, int CH, bool SWIGLU, typename L>
__device__ __forceinline__ void consume_group(uint32_t code_j, uint32_t scale_j, uint32_t fr,
                                              int w, Acc<CH, NB>& acc) {
  constexpr int kTerms = ModeInfo<MODE, NB>::kTerms;
  const float zq[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  uint4 bf[MODE == kN2 ? 1 : NB * kTerms];
#pragma unroll
  for (int i = 0; i < (MODE == kN2 ? 1 : NB * kTerms); ++i) bf[i] = lds128(fr + i * 512);
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int slot = tile_slot<W, CH, SWIGLU>(w, c);
    const uint4 wq = lds128(code_j + slot * L::kCodeTile);
    const uint4 su = lds128(scale_j + slot * L::kScaleTile);
    const float s[4] = {__uint_as_float(su.x), __uint_as_float(su.y), __uint_as_float(su.z),
                        __uint_as_float(su.w)};
#pragma unroll
    for (int T = 0; T < 2; ++T) {
      uint32_t a0[4], a1[4];
      mma::unpack_pair(T ? wq.z : wq.x, T ? wq.w : wq.y, a0, a1);
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        float d[4];
        if constexpr (MODE == kN2) {
          mma::mma_f16_zc(d, a0, bf[0].x, bf[0].y, zq);
          mma::mma_f16(d, a1, bf[0].z, bf[0].w);
        } else {
          const uint4 hi = bf[b * kTerms];
          mma::mma_f16_zc(d, a0, hi.x, hi.y, zq);
          mma::mma_f16(d, a1, hi.z, hi.w);
          if constexpr (kTerms == 2) {
            const uint4 lo = bf[b * kTerms + 1];
            mma::mma_f16(d, a0, lo.x, lo.y);
            mma::mma_f16(d, a1, lo.z, lo.w);
          }
        }
        float(&a)[4] = acc.v[c][T][b];
        a[0] = fmaf(s[2 * T], d[0], a[0]);
        a[1] = fmaf(s[2 * T], d[1], a[1]);
        a[2] = fmaf(s[2 * T + 1], d[2], a[2]);
        a[3] = fmaf(s[2 * T + 1], d[3], a[3]);
      }
    }
  }
}

// Finished outputs of the lane: row `row` (of the slice) of tile c, columns 4h .. 4h + 3, for
// the n-th row this lane holds (kN2: one row, t; otherwise rows 8b + 2t + odd). The row's final
// exponent factor is applied here.
template <int MODE, int CH, int NB>
__device__ __forceinline__ float4 lane_result(const Acc<CH, NB>& acc, int c, int b, int odd,
                                              float f) {
  if constexpr (MODE == kN2) {
    return make_float4(f * (acc.v[c][0][0][0] + acc.v[c][0][0][1]),
                       f * (acc.v[c][0][0][2] + acc.v[c][0][0][3]),
                       f * (acc.v[c][1][0][0] + acc.v[c][1][0][1]),
                       f * (acc.v[c][1][0][2] + acc.v[c][1][0][3]));
  } else {
    return make_float4(f * acc.v[c][0][b][odd], f * acc.v[c][0][b][2 + odd],
                       f * acc.v[c][1][b][odd], f * acc.v[c][1][b][2 + odd]);
  }
}

// ------------------------------------------------------------------------------ producer

// Weight operands of one launch: the fast form copies all of a CTA's tiles of a stage with one
// 4-D (plain) or 5-D (gate/up halves) box, the last coordinate selecting the matrix (an expert
// of stacked MoE weights; 0 for a dense GEMM); the fallback (N or N/2 not a multiple of 32)
// copies one 32-column 3-D box per tile, with columns past the matrix read as zero.
struct WeightMaps {
  CUtensorMap codes, scales;
  int fast;  // 1: multi-tile boxes; 0: per-tile boxes
};

template <int W, int CH, int G, bool SWIGLU, typename L>
__device__ __forceinline__ void issue_stage(const WeightMaps& wm, uint32_t code_dst,
                                            uint32_t scale_dst, uint32_t bar, int q, int cta_tile,
                                            int N, int z) {
  constexpr int kT = L::kTiles;
  mbar_expect_tx(bar, L::kStageTx);
  if (wm.fast) {
    if constexpr (SWIGLU) {
      tma_load_5d(code_dst, &wm.codes, 0, 4 * q, cta_tile * (kT / 2), 0, z, bar);
      tma_load_5d(scale_dst, &wm.scales, 0, q, cta_tile * (kT / 2), 0, z, bar);
    } else {
      tma_load_4d(code_dst, &wm.codes, 0, 4 * q, cta_tile * kT, z, bar);
      tma_load_4d(scale_dst, &wm.scales, 0, q, cta_tile * kT, z, bar);
    }
  } else {
#pragma unroll 1
    for (int i = 0; i < kT; ++i) {
      int col;
      if constexpr (SWIGLU) {
        constexpr int TT = kT / 2;
        col = i < TT ? 32 * (cta_tile * TT + i) : (N >> 1) + 32 * (cta_tile * TT + i - TT);
      } else {
        col = 32 * (cta_tile * kT + i);
      }
      tma_load_3d(code_dst + i * L::kCodeTile, &wm.codes, col, 4 * q, z, bar);
      tma_load_3d(scale_dst + i * L::kScaleTile, &wm.scales, col, q, z, bar);
    }
  }
}

// ------------------------------------------------------------------------------ roles

// Barrier addresses of a CTA (see WsGeo).
template <typename L>
struct Bars {
  uint32_t full, empty, xfull, ffull, fempty, recv;
  __device__ __forceinline__ explicit Bars(char* base) {
    full = smem_u32(base + L::kBarOff);
    empty = full + L::kR * 8;
    xfull = empty + L::kR * 8;
    ffull = xfull + 16;
    fempty = ffull + 16;
    recv = fempty + 16;
  }
};

// Thread 0 initializes every barrier and clears the abort flag; the caller synchronizes the CTA
// afterwards.
template <typename L>
__device__ __forceinline__ void init_roles(char* base) {
  if (threadIdx.x == 0) {
    const Bars<L> b(base);
    for (int i = 0; i < L::kR; ++i) {
      mbar_init(b.full + 8 * i, 1);
      mbar_init(b.empty + 8 * i, L::kConsumers);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(b.xfull + 8 * i, 1);
      mbar_init(b.ffull + 8 * i, 32);
      mbar_init(b.fempty + 8 * i, L::kConsumers);
    }
    mbar_init(b.recv, 1);
    *reinterpret_cast<volatile int*>(base + L::kAbortOff) = 0;
    mma::mbar_fence_init();
  }
}

// Producer (one lane): streams the stages of groups [q0, q0 + nq) of the CTA's tiles. Before it
// returns, every copy it issued has landed (so shared memory can be reused or released).
template <bool SWIGLU, typename L>
__device__ __forceinline__ void producer_loop(const WeightMaps& wm, char* base, int q0, int nq,
                                              int cta_tile, int N, int wz, unsigned int* err) {
  constexpr int R = L::kR, G = L::kG;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + L::kAbortOff);
  const Bars<L> bars(base);
  const uint32_t codes = smem_u32(base + L::kCodeOff), scales = smem_u32(base + L::kScaleOff);
  const int nst = (nq + G - 1) / G;
  int st = 0, issued = 0;
  uint32_t ph = 0;
  for (int s = 0; s < nst; ++s) {
    if (s >= R && !wait_phase(bars.empty + 8 * st, ph ^ 1, abort_flag)) {
      raise_abort(abort_flag, err);
      break;
    }
    issue_stage<L::kW, L::kCH, G, SWIGLU, L>(wm, codes + st * L::kCodeStage,
                                              scales + st * L::kScaleStage, bars.full + 8 * st,
                                              q0 + s * G, cta_tile, N, wz);
    issued = s + 1;
    if (++st == R) {
      st = 0;
      ph ^= 1;
    }
  }
  for (int s = issued > R ? issued - R : 0; s < issued; ++s)
    (void)mma::mbar_wait(bars.full + 8 * (s % R), (s / R) & 1, kWaitLimitNs / 16);
}

// Prep warp: activation chunks [q0 + c CG, ...) -> B fragments (see prep_chunk).
template <typename XT, typename L>
__device__ __forceinline__ void prep_loop(const CUtensorMap* xmap, char* base, int q0, int nq,
                                          int xrow0, unsigned int* err) {
  constexpr int CG = L::kCG;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + L::kAbortOff);
  const Bars<L> bars(base);
  const uint32_t xraw = smem_u32(base + L::kXRawOff);
  const int nch = (nq + CG - 1) / CG;
  int eprev[L::kMode == kN2 ? 1 : L::kNB] = {};
  int issued = nch < 2 ? nch : 2;
  if (lane == 0) {
    dependency_wait();  // the activations may be the previous kernel's output
    for (int c = 0; c < issued; ++c) {
      mbar_expect_tx(bars.xfull + 8 * c, L::kXRawBytes);
      tma_load_2d(xraw + c * L::kXRawBytes, xmap, 32 * (q0 + c * CG), xrow0, bars.xfull + 8 * c);
    }
  }
  for (int c = 0; c < nch; ++c) {
    const int b = c & 1;
    const uint32_t par = (c >> 1) & 1;
    bool ok = wait_phase(bars.xfull + 8 * b, par, abort_flag);
    if (ok && c >= 2) ok = wait_phase(bars.fempty + 8 * b, par ^ 1, abort_flag);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) raise_abort(abort_flag, err);
      break;
    }
    const int ngr = nq - c * CG < CG ? nq - c * CG : CG;
    prep_chunk<L::kMode, L::kNB, XT, L>(base, b, ngr, eprev, c == 0);
    mbar_arrive(bars.ffull + 8 * b);
    fence_proxy_async_smem();  // this lane's reads of the raw chunk precede its next TMA refill
    __syncwarp();
    if (lane == 0 && c + 2 < nch) {
      mbar_expect_tx(bars.xfull + 8 * b, L::kXRawBytes);
      tma_load_2d(xraw + b * L::kXRawBytes, xmap, 32 * (q0 + (c + 2) * CG), xrow0,
                  bars.xfull + 8 * b);
      issued = c + 3;
    }
  }
  if (lane == 0) {
    for (int c = issued > 2 ? issued - 2 : 0; c < issued; ++c)
      (void)mma::mbar_wait(bars.xfull + 8 * (c & 1), (c >> 1) & 1, kWaitLimitNs / 16);
  }
}

// Groups of a stage a consumer warp works on at once: 1 keeps one group's operands in registers
// (more warps fit per SM), G lets the compiler overlap the groups' loads.
#ifndef W4A16_GROUP_UNROLL
#define W4A16_GROUP_UNROLL 2
#endif
constexpr int kGroupUnroll = W4A16_GROUP_UNROLL;

// Offset of lane (g, t)'s 16-byte chunk h of packed row 4j + t in a tile (128-byte swizzle:
// chunk index XOR row % 8).
__device__ __forceinline__ uint32_t code_offset(int j, int t, int h) {
  const int r = 4 * j + t;
  return (uint32_t)(r * 128 + ((h ^ (r & 7)) << 4));
}

// Rows (of the CTA's row slice) held by a consumer lane: kN2 one row (t); otherwise rows
// 8b + 2t + odd, indexed 2b + odd.
template <int MODE, int NB>
struct LaneRows {
  static constexpr int kN = MODE == kN2 ? 1 : 2 * NB;
  __device__ __forceinline__ static int row(int t, int i) {
    return MODE == kN2 ? t : 8 * (i >> 1) + 2 * t + (i & 1);
  }
};

// Consumer warp w: accumulates its tiles over groups [q0, q0 + nq). On return `ex` holds the
// exponent of each of the lane's rows in the last chunk (the accumulators are in units of
// 2^(ex - 14)). Returns false if a wait gave up.
template <bool SWIGLU, typename L>
__device__ __forceinline__ bool consumer_loop(char* base, int nq, int w, unsigned int* err,
                                              Acc<L::kCH, L::kNB>& acc,
                                              int (&ex)[LaneRows<L::kMode, L::kNB>::kN]) {
  constexpr int MODE = L::kMode, NB = L::kNB, W = L::kW, CH = L::kCH, G = L::kG, R = L::kR,
                CG = L::kCG;
  using LR = LaneRows<MODE, NB>;
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base + L::kAbortOff);
  const Bars<L> bars(base);
#pragma unroll
  for (int c = 0; c < CH; ++c)
#pragma unroll
    for (int T = 0; T < 2; ++T)
#pragma unroll
      for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc.v[c][T][b][r] = 0.0f;
#pragma unroll
  for (int i = 0; i < LR::kN; ++i) ex[i] = 0;

  const int h = mma::lane_chunk(g);
  const uint32_t codes = smem_u32(base + L::kCodeOff);
  const uint32_t scales = smem_u32(base + L::kScaleOff) + h * 16;
  const uint32_t frag = smem_u32(base + L::kFragOff) + lane * 16;
  const int* fexp = reinterpret_cast<const int*>(base + L::kExpOff);

  const int nch = (nq + CG - 1) / CG;
  int st = 0;
  uint32_t ph = 0;
  bool ok = true;
  for (int c = 0; c < nch && ok; ++c) {
    const int b = c & 1;
    ok = wait_phase(bars.ffull + 8 * b, (c >> 1) & 1, abort_flag);
    if (!__all_sync(0xffffffffu, ok)) {
      ok = false;
      break;
    }
    int en[LR::kN];
    const bool changed = c == 0 || fexp[L::kExpInts * b + L::kExpFlag] != 0;  // whole warp
#pragma unroll
    for (int i = 0; i < LR::kN; ++i) en[i] = changed ? fexp[L::kExpInts * b + LR::row(t, i)] : ex[i];
    if (c > 0 && changed) {
      // accumulators from chunk units 2^(ex - 14) to 2^(en - 14)
#pragma unroll
      for (int i = 0; i < LR::kN; ++i) {
        const int d = ex[i] - en[i];
        const float f = mma::exp2i(d >> 1) * mma::exp2i(d - (d >> 1));
        const int bb = MODE == kN2 ? 0 : (i >> 1), odd = i & 1;
#pragma unroll
        for (int cc = 0; cc < CH; ++cc)
#pragma unroll
          for (int T = 0; T < 2; ++T) {
            if constexpr (MODE == kN2) {
#pragma unroll
              for (int r = 0; r < 4; ++r) acc.v[cc][T][0][r] *= f;
            } else {
              acc.v[cc][T][bb][odd] *= f;
              acc.v[cc][T][bb][odd + 2] *= f;
            }
          }
      }
    }
#pragma unroll
    for (int i = 0; i < LR::kN; ++i) ex[i] = en[i];
    const int ngr = nq - c * CG < CG ? nq - c * CG : CG;
    const uint32_t fr = frag + b * L::kFragBytes;
    for (int q = 0; q < ngr; q += G) {
      if (!wait_consumer(bars.full + 8 * st, ph, abort_flag)) ok = false;
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      const uint32_t cs = codes + st * L::kCodeStage, ss = scales + st * L::kScaleStage;
#pragma unroll(kGroupUnroll)
      for (int j = 0; j < G; ++j) {
        if (q + j < ngr)
          consume_group<MODE, NB, W, CH, SWIGLU, L>(cs + code_offset(j, t, h), ss + j * 128,
                                                    fr + (q + j) * ModeInfo<MODE, NB>::kFragGroup,
                                                    w, acc);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.empty + 8 * st);
      if (++st == R) {
        st = 0;
        ph ^= 1;
      }
    }
    __syncwarp();
    if (ok && lane == 0) mbar_arrive(bars.fempty + 8 * b);
  }
  if (!ok && lane == 0) raise_abort(abort_flag, err);
  return ok;
}

}  // namespace ws
}  // namespace w4a16
