// Tensor-core weight-streaming core for small M (decode / draft-tree verify).
//
// Each warp owns a slice of 32*CH weight columns and walks the CTA's K range two groups
// (2 x 32 k) per pipeline stage. Per stage it:
//   * receives, by TMA (one elected lane issues 2*CH tile copies into the warp's ring of R
//     stages, 2 to 4 by geometry, with an mbarrier per stage), CH tiles of 32 columns x 8 packed
//     rows of the codes (128-byte swizzle, so the lanes' 16-byte reads below are bank-conflict
//     free) and CH tiles of 32 columns x 2 rows of the scales;
//   * turns each lane's 4 words per tile into fp16 MMA A-fragments with two bit tricks:
//     (w & 0x000F000F) | 0x64006400 is the fp16 pair (1024 + nibble_0, 1024 + nibble_4), and the
//     same mask shifted by 4 gives 1024 + 16 * nibble; one fp16 FMA then yields nibble - 8;
//   * multiplies them with the activations on the tensor cores (mma.sync m16n8k16, fp16 in,
//     fp32 accumulate) -- the activations enter as two fp16 terms, x * 2^-e = hi + lo with a
//     per-group power-of-two e, which carries 22 significant bits of each float32 activation;
//   * applies the group scale times 2^e to the fresh fp32 group sums with one FMA each.
// The unpacked codes are exact integers, products of codes and fp16 terms are exact in fp32,
// so the only rounding beyond float32 accumulation is the ~2^-22 relative cut of x.
// A bf16 mode (stream_groups<..., B16 = true>) serves bf16 activations: the codes unpack to
// bf16 instead, and the activations are MMA operands as they are (no split, no exponent).
//
// MMA operand mapping (m16n8k16; g = lane / 4, t = lane % 4):
//   A (16 x 16): rows = weight columns, k = input index. Lane (g, t) holds the packed word of
//     row 4q + t of the group q for two columns (A rows g and g + 8). Within the group, MMA
//     k-slot 2t + {0, 1} is input 8t + {0, 4} (k-step 0, register a0/a1), slot 2t + 8 + {0, 1}
//     is 8t + {1, 5}; k-step 1 uses 8t + {2, 6} and 8t + {3, 7}. Any fixed permutation of k
//     inside a group is allowed because the reduction over k does not care about order.
//   B (16 x 8): columns = (row m of x, term): column c of block b is m = 4b + c / 2, term c % 2.
//     Lane (g, t) therefore needs x terms at inputs 8t .. 8t + 7 of one row and term, stored
//     pre-permuted as (0, 4, 1, 5, 2, 6, 3, 7) so that one 16-byte shared load gives b0/b1 of
//     both k-steps.
//   C (16 x 8): lane (g, t) ends with row m = 4b + t, terms hi/lo, for its two A rows.
// Chunk mapping: in each 32-column tile lane (g, t) owns the 16-byte chunk h(g) = g/2 + 4 (g%2),
//   i.e. columns 4 h .. 4 h + 3; A tile T (0, 1) uses columns 4h + 2T (row g) and 4h + 2T + 1
//   (row g + 8). With the 128-byte swizzle (16-byte chunk index XOR row % 8) the 8 lanes of
//   each quarter-warp then hit 8 different bank groups.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace w4a16 {
namespace mma {

constexpr int kXChunkBytes = 512;  // activation fragments per (group, n8 block): 32 lanes x 16 B

// ------------------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ float lds32f(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];\n" : "=f"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
               : "memory");
}
// One bounded wait step: the thread sleeps until phase `parity` of the barrier completes or
// about `hint_ns` pass (no busy spinning), and reports whether the phase completed.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
  return t;
}
// Waits for phase `parity` of the barrier, sleeping in steps of at most 1 ms; gives up once
// `limit_ns` of wall time have passed and returns false. The clock is read only after a
// step that ended without the phase completing.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  constexpr uint32_t kStepNs = 1000000u;
  if (mbar_try_wait(bar, parity, kStepNs)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity, kStepNs)) {
    if (global_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// As mbar_wait, but polls with try_wait without a sleep hint (the hardware's own short
// suspend), for hand-offs between warps of one CTA that recur every few hundred nanoseconds.
__device__ __forceinline__ bool mbar_try_wait_poll(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_poll(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait_poll(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait_poll(bar, parity)) {
    if (global_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// Cluster forms: this CTA's rank, the cluster address of a shared variable in CTA `rank`, an
// arrive on a (possibly remote) barrier with cluster-scope release, a polled wait with
// cluster-scope acquire (for barriers that other CTAs' threads arrive on), and a full cluster
// barrier.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];\n" ::"r"(cluster_addr)
               : "memory");
}
// Release of this CTA's shared-memory writes at cluster scope (cheaper than a full release: only
// shared::cta accesses are ordered), to pair with mbar_arrive_remote_relaxed.
__device__ __forceinline__ void fence_release_shared_cluster() {
  asm volatile("fence.release.sync_restrict::shared::cta.cluster;\n" ::: "memory");
}
// Acquire counterpart: later accesses to the cluster's shared memory are ordered after a
// completed barrier wait.
__device__ __forceinline__ void fence_acquire_shared_cluster() {
  asm volatile("fence.acquire.sync_restrict::shared::cluster.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];\n" ::"r"(cluster_addr)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (global_ns() - t0 > limit_ns) return false;
  }
  return true;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::
                   : "memory");
}

// TMA tile copy of a 3-D tensor into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Tensor-core product with the accumulator input taken from a loop-invariant zero quad.
__device__ __forceinline__ void mma_f16_zc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                           uint32_t b1, const float (&z)[4]) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%11,%12,%13};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z[0]), "f"(z[1]),
        "f"(z[2]), "f"(z[3]));
}

// (a & mask) | 0x64006400 in one LOP3.
__device__ __forceinline__ uint32_t lop_and_or(uint32_t a, uint32_t mask) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;\n" : "=r"(r) : "r"(a), "r"(mask), "r"(0x64006400u));
  return r;
}

__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;\n" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// Word -> four fp16x2 registers of (nibble - 8):
//   p[0] = (n0, n4), p[1] = (n1, n5), p[2] = (n2, n6), p[3] = (n3, n7).
__device__ __forceinline__ void unpack_word(uint32_t w, uint32_t (&p)[4]) {
  const uint32_t ONE = 0x3C003C00u;        // (1.0, 1.0)
  const uint32_t SIXTEENTH = 0x2C002C00u;  // (1/16, 1/16)
  const uint32_t M1032 = 0xE408E408u;      // (-1032, -1032)
  const uint32_t M72 = 0xD480D480u;        // (-72, -72)
  const uint32_t w8 = w >> 8;
  p[0] = hfma2_u32(lop_and_or(w, 0x000F000Fu), ONE, M1032);
  p[1] = hfma2_u32(lop_and_or(w, 0x00F000F0u), SIXTEENTH, M72);
  p[2] = hfma2_u32(lop_and_or(w8, 0x000F000Fu), ONE, M1032);
  p[3] = hfma2_u32(lop_and_or(w8, 0x00F000F0u), SIXTEENTH, M72);
}

// Two words (columns of A rows g and g + 8) -> the A fragments of both k-steps, written in
// operand order so no register moves are needed:
//   a0 = (n0 n4 of wa, n0 n4 of wb, n1 n5 of wa, n1 n5 of wb), a1 = the same for n2 n6 / n3 n7.
__device__ __forceinline__ void unpack_pair(uint32_t wa, uint32_t wb, uint32_t (&a0)[4],
                                            uint32_t (&a1)[4]) {
  const uint32_t ONE = 0x3C003C00u, SIXTEENTH = 0x2C002C00u;
  const uint32_t M1032 = 0xE408E408u, M72 = 0xD480D480u;
  const uint32_t wa8 = wa >> 8, wb8 = wb >> 8;
  a0[0] = hfma2_u32(lop_and_or(wa, 0x000F000Fu), ONE, M1032);
  a0[1] = hfma2_u32(lop_and_or(wb, 0x000F000Fu), ONE, M1032);
  a0[2] = hfma2_u32(lop_and_or(wa, 0x00F000F0u), SIXTEENTH, M72);
  a0[3] = hfma2_u32(lop_and_or(wb, 0x00F000F0u), SIXTEENTH, M72);
  a1[0] = hfma2_u32(lop_and_or(wa8, 0x000F000Fu), ONE, M1032);
  a1[1] = hfma2_u32(lop_and_or(wb8, 0x000F000Fu), ONE, M1032);
  a1[2] = hfma2_u32(lop_and_or(wa8, 0x00F000F0u), SIXTEENTH, M72);
  a1[3] = hfma2_u32(lop_and_or(wb8, 0x00F000F0u), SIXTEENTH, M72);
}

// bf16 forms for activations that arrive in bf16: A and B of one MMA share their type, so the
// codes are unpacked to bf16 instead. ((w >> 4j) & 0x000F000F) | 0x43004300 is the bf16 pair
// (128 + n_j, 128 + n_{j+4}); one bf16 FMA subtracts 136 exactly. Same register order as
// unpack_pair.
__device__ __forceinline__ uint32_t bfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;\n" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}
__device__ __forceinline__ uint32_t lop_and_or_b16(uint32_t a) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;\n" : "=r"(r) : "r"(a), "r"(0x000F000Fu), "r"(0x43004300u));
  return r;
}
__device__ __forceinline__ void unpack_pair_b16(uint32_t wa, uint32_t wb, uint32_t (&a0)[4],
                                                uint32_t (&a1)[4]) {
  const uint32_t ONE = 0x3F803F80u, M136 = 0xC308C308u;  // bf16 (1, 1), (-136, -136)
  a0[0] = bfma2_u32(lop_and_or_b16(wa), ONE, M136);
  a0[1] = bfma2_u32(lop_and_or_b16(wb), ONE, M136);
  a0[2] = bfma2_u32(lop_and_or_b16(wa >> 4), ONE, M136);
  a0[3] = bfma2_u32(lop_and_or_b16(wb >> 4), ONE, M136);
  a1[0] = bfma2_u32(lop_and_or_b16(wa >> 8), ONE, M136);
  a1[1] = bfma2_u32(lop_and_or_b16(wb >> 8), ONE, M136);
  a1[2] = bfma2_u32(lop_and_or_b16(wa >> 12), ONE, M136);
  a1[3] = bfma2_u32(lop_and_or_b16(wb >> 12), ONE, M136);
}
__device__ __forceinline__ void mma_b16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_b16_zc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                           uint32_t b1, const float (&z)[4]) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%10,%11,%12,%13};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z[0]), "f"(z[1]),
        "f"(z[2]), "f"(z[3]));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Exact power of two 2^e for e in [-126, 127].
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((e + 127) << 23); }

// ------------------------------------------------------------------------------ activations

// Preparing the B fragments of one group q (inputs 32q .. 32q + 31) for rows 0 .. M-1 (rows
// >= M are zero) takes two steps so the loads can be issued long before their use:
//   prep_load : lane (g, t) loads x[m][32q + 8t .. +7] for m = 4b + g/2 into registers;
//   prep_store: the warp finds the group's largest magnitude, scales by 2^-e, splits into fp16
//               hi/lo terms and writes NB x 512 B at dst plus the group's 2^e at *fscale.
// rowptr(m) returns a pointer to row m of x (float32, 16-byte aligned).
template <int NB, typename RowPtr>
__device__ __forceinline__ void prep_load(const RowPtr& rowptr, int M, int q, float (&v)[NB][8]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const int m = 4 * b + (g >> 1);
    if (m < M) {
      const float4* p = reinterpret_cast<const float4*>(rowptr(m) + 32 * q + 8 * t);
      const float4 u0 = __ldg(p), u1 = __ldg(p + 1);
      v[b][0] = u0.x; v[b][1] = u0.y; v[b][2] = u0.z; v[b][3] = u0.w;
      v[b][4] = u1.x; v[b][5] = u1.y; v[b][6] = u1.z; v[b][7] = u1.w;
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[b][j] = 0.0f;
    }
  }
}

// Power-of-two exponent e of a group: its largest magnitude times 2^-e lies in [2^14, 2^15),
// far from fp16 overflow (65504) and with the lo term of every element within 2^17 of it
// still a normal fp16 number. (Warp-wide: every lane passes its own partial maximum.)
__device__ __forceinline__ int group_exponent(float amax) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  int ex = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127;
  if (amax == 0.0f) ex = 0;
  return ex < -110 ? -110 : (ex > 110 ? 110 : ex);
}

template <int NB>
__device__ __forceinline__ void prep_store(const float (&v)[NB][8], char* dst, float* fscale) {
  const int lane = threadIdx.x & 31, g = lane >> 2;
  float amax = 0.0f;
#pragma unroll
  for (int b = 0; b < NB; ++b)
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[b][j]));
  const int ex = group_exponent(amax);
  const float up = exp2i(14 - ex);
  const bool lo_term = (g & 1) != 0;
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    float o[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float xs = v[b][j] * up;
      const float hi = __half2float(__float2half_rn(xs));
      o[j] = lo_term ? (xs - hi) : xs;
    }
    uint4 r;
    r.x = pack_half2(o[0], o[4]);
    r.y = pack_half2(o[1], o[5]);
    r.z = pack_half2(o[2], o[6]);
    r.w = pack_half2(o[3], o[7]);
    *reinterpret_cast<uint4*>(dst + b * kXChunkBytes + lane * 16) = r;
  }
  if (lane == 0) *fscale = exp2i(ex - 14);
}

// Activations in bf16: no split is needed (an MMA column is one row m = 8b + g of x, the
// product of a bf16 activation and an exact code is exact in fp32) and no exponent (fscale = 1).
// prep_load_b16: lane (g, t) loads x[m][32q + 8t .. +7] (16 bytes) for m = 8b + g;
// prep_store_b16: byte permutes put the 8 values in the k order of the codes
// (0, 4, 1, 5, 2, 6, 3, 7) and write NB x 512 B at dst.
template <int NB, bool B16>
struct PrepRegs {
  float v[NB][8];
};
template <int NB>
struct PrepRegs<NB, true> {
  uint4 v[NB];
};

template <int NB, typename RowPtr>
__device__ __forceinline__ void prep_load_b16(const RowPtr& rowptr, int M, int q, uint4 (&v)[NB]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const int m = 8 * b + g;
    v[b] = m < M ? __ldg(reinterpret_cast<const uint4*>(rowptr(m) + 32 * q + 8 * t))
                 : make_uint4(0u, 0u, 0u, 0u);
  }
}
template <int NB>
__device__ __forceinline__ void prep_store_b16(const uint4 (&v)[NB], char* dst, float* fscale) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    uint4 r;
    r.x = __byte_perm(v[b].x, v[b].z, 0x5410);  // k 0, 4
    r.y = __byte_perm(v[b].x, v[b].z, 0x7632);  // k 1, 5
    r.z = __byte_perm(v[b].y, v[b].w, 0x5410);  // k 2, 6
    r.w = __byte_perm(v[b].y, v[b].w, 0x7632);  // k 3, 7
    *reinterpret_cast<uint4*>(dst + b * kXChunkBytes + lane * 16) = r;
  }
  if (lane == 0) *fscale = 1.0f;
}

template <int NB, bool B16, typename RowPtr>
__device__ __forceinline__ void prep_load_any(const RowPtr& rowptr, int M, int q,
                                              PrepRegs<NB, B16>& r) {
  if constexpr (B16) prep_load_b16<NB>(rowptr, M, q, r.v);
  else prep_load<NB>(rowptr, M, q, r.v);
}
template <int NB, bool B16>
__device__ __forceinline__ void prep_store_any(const PrepRegs<NB, B16>& r, char* dst,
                                               float* fscale) {
  if constexpr (B16) prep_store_b16<NB>(r.v, dst, fscale);
  else prep_store<NB>(r.v, dst, fscale);
}

// ------------------------------------------------------------------------------ geometry

constexpr int kRows = 8;     // packed rows per stage (2 groups)

#ifndef W4A16_UNROLL_GROUPS
#define W4A16_UNROLL_GROUPS 2
#endif
constexpr int kUnrollGroups = W4A16_UNROLL_GROUPS;  // groups of a stage interleaved by the compiler
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // give up a barrier wait after 2 s

// Shared-memory layout of one CTA (offsets from a 1024-byte aligned base). Everything up to
// the x region depends only on CH and WN, so kernels that switch NB per job share barriers:
//   codes   WN x R x CH tiles of 8 x 128 B (swizzled)
//   scales  WN x R x CH tiles of 2 x 128 B
//   bars    WN x R mbarriers (padded to 128 B)
//   x       activation fragments: the CTA's whole K range when it fits in XB bytes, else two
//           alternating halves
//   fscale  2^e per prepared group
// R = stages per warp ring, XB = activation-fragment budget.
template <int NB, int CH, int WN, int R, int XB>
struct Geo {
  static constexpr int kRing = R;
  static constexpr int kCodeTile = kRows * 128;
  static constexpr int kScaleTile = (kRows / 4) * 128;
  static constexpr int kCodeOff = 0;
  static constexpr int kScaleOff = kCodeOff + WN * kRing * CH * kCodeTile;
  static constexpr int kBarOff = kScaleOff + WN * kRing * CH * kScaleTile;
  static constexpr int kXOff = kBarOff + ((WN * kRing * 8 + 127) / 128) * 128;
  static constexpr int kXGroups = (XB / (NB * kXChunkBytes)) & ~1;
  static constexpr int kFOff = kXOff + kXGroups * NB * kXChunkBytes;
  static constexpr int kBytes = kFOff + ((kXGroups * 4 + 127) / 128) * 128;
  static constexpr int kAlloc = kBytes + 1024;  // room to align the base
  static constexpr uint32_t kStageTx = CH * (kCodeTile + kScaleTile);
};

// First 1024-byte aligned address (in the shared window) at or after p.
__device__ __forceinline__ char* align1024(char* p) {
  const uint32_t s = smem_u32(p);
  return p + ((1024u - (s & 1023u)) & 1023u);
}

__device__ __forceinline__ int lane_chunk(int g) { return (g >> 1) + 4 * (g & 1); }

// Tensor column of the 32-column tile c of slice s.
//   plain         : 32 CH s + 32 c.
//   SwiGLU (CH>=2): tiles c < CH/2 are gate columns 16 CH s + 32 c; tiles c >= CH/2 the
//                   matching up columns I + 16 CH s + 32 (c - CH/2).
template <int CH, bool SWIGLU>
__device__ __forceinline__ int tile_x(int slice, int c, int N) {
  if (SWIGLU) {
    constexpr int H = CH / 2;
    const int j = 32 * H * slice + 32 * (c >= H ? c - H : c);
    return c >= H ? (N >> 1) + j : j;
  }
  return 32 * CH * slice + 32 * c;
}

// Output position of the lane's 4 columns of tile c: plain -> weight column (valid if < N);
// SwiGLU -> output index j of gate tile c (valid if < I).
template <int CH, bool SWIGLU>
__device__ __forceinline__ int out_col(int slice, int c, int g, int N, bool* valid) {
  if (SWIGLU) {
    constexpr int H = CH / 2;
    const int j = 32 * H * slice + 32 * c + 4 * lane_chunk(g);
    *valid = j < (N >> 1);
    return j;
  }
  const int col = 32 * CH * slice + 32 * c + 4 * lane_chunk(g);
  *valid = col < N;
  return col;
}

// ------------------------------------------------------------------------------ main loop

// Initializes this warp's stage barriers (once per kernel, before the first stream_groups).
template <typename L>
__device__ __forceinline__ void init_barriers(char* base, int warps) {
  constexpr int kRing = L::kRing;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  (void)warps;
  if (lane == 0) {
    const uint32_t bar_s = smem_u32(base + L::kBarOff) + warp * kRing * 8;
    for (int i = 0; i < kRing; ++i) mbar_init(bar_s + i * 8, 1);
    mbar_fence_init();
  }
  __syncwarp();
}

// The CTA's warps stream groups q0 .. q0 + nq - 1 of their slices (slice = slice0 + warp) of
// matrix `z` of the descriptors, accumulating acc[c][T][b][r] (tile c, A tile T, n8 block b,
// C register r). `seq` counts the stages this warp has used so far (barrier phases carry on
// across calls). Returns false if a barrier wait gave up (the error word is then set).
// All threads of the CTA must call this (it synchronizes the CTA around the x fragments).
template <int NB, int CH, bool SWIGLU, int WN, typename L, bool B16 = false, typename RowPtr>
__device__ __forceinline__ bool stream_groups(const RowPtr& rowptr, int M,
                                              const CUtensorMap* tq, const CUtensorMap* ts,
                                              int z, int N, int q0, int nq, int slice0,
                                              char* base, int& seq, unsigned int* err,
                                              float (&acc)[CH][2][NB][4]) {
  static_assert(!SWIGLU || CH >= 2, "fused SwiGLU tiles pair gate and up tiles");
  constexpr int kRing = L::kRing;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int slice = slice0 + warp;
  const uint32_t code_s = smem_u32(base + L::kCodeOff) + warp * kRing * CH * L::kCodeTile;
  const uint32_t scale_s = smem_u32(base + L::kScaleOff) + warp * kRing * CH * L::kScaleTile;
  const uint32_t bar_s = smem_u32(base + L::kBarOff) + warp * kRing * 8;
  char* xbuf = base + L::kXOff;
  float* fsc = reinterpret_cast<float*>(base + L::kFOff);

  // Is any column of this warp's slice inside the matrix? (Its first columns are.)
  bool any;
  out_col<CH, SWIGLU>(slice, 0, 0, N, &any);

#pragma unroll
  for (int c = 0; c < CH; ++c)
#pragma unroll
    for (int T = 0; T < 2; ++T)
#pragma unroll
      for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int r = 0; r < 4; ++r) acc[c][T][b][r] = 0.0f;

  const int nst = (nq + 1) >> 1;  // stages of 2 groups (the last may hold 1)
  auto issue = [&](int s) {       // lane 0 only
    const int u = seq + s;
    const int st = u % kRing;
    const uint32_t bar = bar_s + st * 8;
    mbar_expect_tx(bar, L::kStageTx);
    const int row = 4 * (q0 + 2 * s);
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int x = tile_x<CH, SWIGLU>(slice, c, N);
      tma_load_3d(code_s + (st * CH + c) * L::kCodeTile, tq, x, row, z, bar);
      tma_load_3d(scale_s + (st * CH + c) * L::kScaleTile, ts, x, q0 + 2 * s, z, bar);
    }
  };
  if (any && lane == 0) {
    for (int s = 0; s < kRing - 1 && s < nst; ++s) issue(s);
  }

  // Activation fragments: the whole range at once when it fits; otherwise chunks of WN groups
  // (one per warp), double-buffered, whose loads are issued before the previous chunk's
  // compute and converted after it.
  static_assert(L::kXGroups >= 2 * WN && WN % 2 == 0, "x region must hold two chunks");
  const int pg = nq <= L::kXGroups ? ((nq + 1) & ~1) : WN;
  for (int j = warp; j < pg; j += WN) {
    if (j < nq) {
      PrepRegs<NB, B16> v;
      prep_load_any<NB, B16>(rowptr, M, q0 + j, v);
      prep_store_any<NB, B16>(v, xbuf + j * NB * kXChunkBytes, &fsc[j]);
    }
  }
  __syncthreads();

  bool ok = true;
  int fail_s = 0;
  const float zq[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  const uint32_t xbuf_s = smem_u32(xbuf) + lane * 16;
  const uint32_t fsc_s = smem_u32(fsc);
  const int h = lane_chunk(g);
  const int nchunks = (nq + pg - 1) / pg;
  const int sps = pg >> 1;  // stages per x chunk
  for (int pc = 0; pc < nchunks; ++pc) {
    const int buf = pc & 1;
    // Next chunk's activations: loads now, conversion after this chunk's compute.
    PrepRegs<NB, B16> nv;
    const int qn = (pc + 1) * pg + warp;
    const bool more = pc + 1 < nchunks && qn < nq;
    if (more) prep_load_any<NB, B16>(rowptr, M, q0 + qn, nv);
    const int s_end = ((pc + 1) * sps < nst) ? (pc + 1) * sps : nst;
    if (any) {
      for (int s = pc * sps; s < s_end; ++s) {
        if (ok && lane == 0 && s + kRing - 1 < nst) issue(s + kRing - 1);
        const int u = seq + s;
        const int st = u % kRing;
        if (ok) {
          const bool got = mbar_wait(bar_s + st * 8, (u / kRing) & 1, kWaitLimitNs);
          if (!__all_sync(0xffffffffu, got)) {  // warp-uniform decision
            ok = false;
            fail_s = s;
            if (lane == 0 && err) atomicCAS(err, 0u, 8u);  // W4A16_ERR_TIMEOUT
          }
        }
        if (ok) {
#pragma unroll (kUnrollGroups)
          for (int j = 0; j < 2; ++j) {
            const int qi = 2 * s + j;
            if (qi < nq) {
              const int r = 4 * j + t;
              const uint32_t coff = r * 128 + ((h ^ (r & 7)) << 4);
              uint4 wq[CH];
              float4 s4[CH];
#pragma unroll
              for (int c = 0; c < CH; ++c) {
                wq[c] = lds128(code_s + (st * CH + c) * L::kCodeTile + coff);
                const uint4 u4 =
                    lds128(scale_s + (st * CH + c) * L::kScaleTile + j * 128 + h * 16);
                s4[c] = make_float4(__uint_as_float(u4.x), __uint_as_float(u4.y),
                                    __uint_as_float(u4.z), __uint_as_float(u4.w));
              }
              const int xi = buf * pg + (qi - pc * pg);
              const float fg = lds32f(fsc_s + xi * 4);
              uint4 bf[NB];
#pragma unroll
              for (int b = 0; b < NB; ++b) bf[b] = lds128(xbuf_s + (xi * NB + b) * kXChunkBytes);
#pragma unroll
              for (int c = 0; c < CH; ++c) {
                const float sv[4] = {s4[c].x * fg, s4[c].y * fg, s4[c].z * fg, s4[c].w * fg};
#pragma unroll
                for (int T = 0; T < 2; ++T) {
                  uint32_t a0[4], a1[4];
                  if constexpr (B16)
                    unpack_pair_b16(T ? wq[c].z : wq[c].x, T ? wq[c].w : wq[c].y, a0, a1);
                  else
                    unpack_pair(T ? wq[c].z : wq[c].x, T ? wq[c].w : wq[c].y, a0, a1);
#pragma unroll
                  for (int b = 0; b < NB; ++b) {
                    float d[4];
                    if constexpr (B16) {
                      mma_b16_zc(d, a0, bf[b].x, bf[b].y, zq);
                      mma_b16(d, a1, bf[b].z, bf[b].w);
                    } else {
                      mma_f16_zc(d, a0, bf[b].x, bf[b].y, zq);
                      mma_f16(d, a1, bf[b].z, bf[b].w);
                    }
                    acc[c][T][b][0] = fmaf(sv[2 * T], d[0], acc[c][T][b][0]);
                    acc[c][T][b][1] = fmaf(sv[2 * T], d[1], acc[c][T][b][1]);
                    acc[c][T][b][2] = fmaf(sv[2 * T + 1], d[2], acc[c][T][b][2]);
                    acc[c][T][b][3] = fmaf(sv[2 * T + 1], d[3], acc[c][T][b][3]);
                  }
                }
              }
            }
          }
        }
        __syncwarp();  // every lane is done with stage st before lane 0 refills it
      }
    }
    if (more)
      prep_store_any<NB, B16>(nv, xbuf + ((buf ^ 1) * pg + warp) * NB * kXChunkBytes,
                              &fsc[(buf ^ 1) * pg + warp]);
    if (nchunks > 1) __syncthreads();
  }
  if (any && !ok) {
    // Let the copies still in flight (stages fail_s .. fail_s + kRing - 2 at most) land before
    // the shared memory is reused or released.
    for (int s = fail_s; s < nst && s < fail_s + kRing; ++s) {
      const int u = seq + s;
      (void)mbar_wait(bar_s + (u % kRing) * 8, (u / kRing) & 1, kWaitLimitNs / 16);
    }
  }
  if (any) seq += nst;  // barrier phases advance only for warps that used them
  __syncthreads();  // the caller may reuse the code ring for its epilogue
  return ok;
}

// ------------------------------------------------------------------------------ epilogues

// Per lane: the 4 finished outputs (hi + lo terms) of row m = 4b + t for tile c.
template <int NB, int CH>
__device__ __forceinline__ float4 chunk_result(const float (&acc)[CH][2][NB][4], int c, int b) {
  return make_float4(acc[c][0][b][0] + acc[c][0][b][1], acc[c][0][b][2] + acc[c][0][b][3],
                     acc[c][1][b][0] + acc[c][1][b][1], acc[c][1][b][2] + acc[c][1][b][3]);
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

__device__ __forceinline__ float4 swiglu4(float4 gt, float4 up) {
  return make_float4(silu_f(gt.x) * up.x, silu_f(gt.y) * up.y, silu_f(gt.z) * up.z,
                     silu_f(gt.w) * up.w);
}

// Writes the lane's finished outputs straight to y (used when one CTA covers the whole K).
// Plain: y[M, N].  SwiGLU: y[M, N/2] = silu(gate) * up (gate tile c pairs with up tile c+CH/2).
template <int NB, int CH, bool SWIGLU>
__device__ __forceinline__ void store_direct(const float (&acc)[CH][2][NB][4], int slice, int N,
                                             int M, float* y) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const int m = 4 * b + t;
    if (m >= M) continue;
    if (SWIGLU) {
      constexpr int H = CH / 2;
      const int I = N >> 1;
#pragma unroll
      for (int c = 0; c < H; ++c) {
        bool valid;
        const int j = out_col<CH, SWIGLU>(slice, c, g, N, &valid);
        if (valid)
          *reinterpret_cast<float4*>(y + (size_t)m * I + j) =
              swiglu4(chunk_result<NB, CH>(acc, c, b), chunk_result<NB, CH>(acc, c + H, b));
      }
    } else {
#pragma unroll
      for (int c = 0; c < CH; ++c) {
        bool valid;
        const int col = out_col<CH, SWIGLU>(slice, c, g, N, &valid);
        if (valid)
          *reinterpret_cast<float4*>(y + (size_t)m * N + col) = chunk_result<NB, CH>(acc, c, b);
      }
    }
  }
}

// Tile-local column of tile c of lane g in a split-K reduction tile (plain: weight column
// within the CTA tile; SwiGLU: gate output index within the tile, with the up values stored
// WN*16*CH columns later).
template <int CH, bool SWIGLU, int WN>
__device__ __forceinline__ int tile_local_col(int warp, int c, int g) {
  const int h4 = 4 * lane_chunk(g);
  if (SWIGLU) {
    constexpr int H = CH / 2;
    constexpr int SO = 16 * CH;  // outputs per slice
    return (c >= H ? WN * SO : 0) + warp * SO + 32 * (c >= H ? c - H : c) + h4;
  }
  return warp * 32 * CH + 32 * c + h4;
}

// ------------------------------------------------------------------------------ 9..16 rows
//
// For 9..16 activation rows the roles swap: A (16 x 16) = activations (rows m = g and g + 8),
// B (16 x 8) = codes, so the hi and lo activation terms are two A operands accumulating into
// the same C and no MMA row is padding. B column n of n8-tile i is weight column 4 h(n) + i of
// the 32-column tile: lane (g, t) loads chunk h(g) (columns 4h .. 4h + 3) of packed row 4q + t,
// and word i of it is its B fragment for n8-tile i (k-slots as in the other orientation).
// C: lane (g, t) holds rows g, g + 8 and B columns 2t, 2t + 1 of each n8-tile i, i.e. weight
// columns 4 h(2t) + i and 4 h(2t + 1) + i.

// Preparing the A fragments of group q for rows 0 .. M-1 (M <= 16; others zero), in two steps
// as for the other orientation. Output: 4 x 512 B at dst, chunk (term * 2 + kstep), each an
// A operand quad in register order: (row g pair 2ks, row g+8 pair 2ks, row g pair 2ks+1,
// row g+8 pair 2ks+1), pair p of a row = inputs (8t + p, 8t + p + 4); term 0 = hi, 1 = lo.
template <typename RowPtr>
__device__ __forceinline__ void prep_load_xa(const RowPtr& rowptr, int M, int q, float (&v)[2][8]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    const int m = g + 8 * hf;
    if (m < M) {
      const float4* p = reinterpret_cast<const float4*>(rowptr(m) + 32 * q + 8 * t);
      const float4 u0 = __ldg(p), u1 = __ldg(p + 1);
      v[hf][0] = u0.x; v[hf][1] = u0.y; v[hf][2] = u0.z; v[hf][3] = u0.w;
      v[hf][4] = u1.x; v[hf][5] = u1.y; v[hf][6] = u1.z; v[hf][7] = u1.w;
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[hf][j] = 0.0f;
    }
  }
}

__device__ __forceinline__ void prep_store_xa(const float (&v)[2][8], char* dst, float* fscale) {
  const int lane = threadIdx.x & 31;
  float amax = 0.0f;
#pragma unroll
  for (int hf = 0; hf < 2; ++hf)
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[hf][j]));
  const int ex = group_exponent(amax);
  const float up = exp2i(14 - ex);
  uint32_t ph[2][4], pl[2][4];  // [half][pair]
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    float hi[8], lo[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float xs = v[hf][j] * up;
      hi[j] = __half2float(__float2half_rn(xs));
      lo[j] = xs - hi[j];
    }
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      ph[hf][p] = pack_half2(hi[p], hi[p + 4]);
      pl[hf][p] = pack_half2(lo[p], lo[p + 4]);
    }
  }
#pragma unroll
  for (int ks = 0; ks < 2; ++ks) {
    *reinterpret_cast<uint4*>(dst + (0 * 2 + ks) * kXChunkBytes + lane * 16) =
        make_uint4(ph[0][2 * ks], ph[1][2 * ks], ph[0][2 * ks + 1], ph[1][2 * ks + 1]);
    *reinterpret_cast<uint4*>(dst + (1 * 2 + ks) * kXChunkBytes + lane * 16) =
        make_uint4(pl[0][2 * ks], pl[1][2 * ks], pl[0][2 * ks + 1], pl[1][2 * ks + 1]);
  }
  if (lane == 0) *fscale = exp2i(ex - 14);
}

// As stream_groups, for 9..16 rows: acc[c][i][r] (tile c, n8-tile i, C register r).
template <int CH, bool SWIGLU, int WN, typename L, typename RowPtr>
__device__ __forceinline__ bool stream_groups_xa(const RowPtr& rowptr, int M,
                                                 const CUtensorMap* tq, const CUtensorMap* ts,
                                                 int z, int N, int q0, int nq, int slice0,
                                                 char* base, int& seq, unsigned int* err,
                                                 float (&acc)[CH][4][4]) {
  static_assert(!SWIGLU || CH >= 2, "fused SwiGLU tiles pair gate and up tiles");
  constexpr int kRing = L::kRing;
  constexpr int kXG = 4 * kXChunkBytes;  // prepared bytes per group
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int slice = slice0 + warp;
  const uint32_t code_s = smem_u32(base + L::kCodeOff) + warp * kRing * CH * L::kCodeTile;
  const uint32_t scale_s = smem_u32(base + L::kScaleOff) + warp * kRing * CH * L::kScaleTile;
  const uint32_t bar_s = smem_u32(base + L::kBarOff) + warp * kRing * 8;
  char* xbuf = base + L::kXOff;
  float* fsc = reinterpret_cast<float*>(base + L::kFOff);
  constexpr int kXGroups = L::kXGroups;  // L is a Geo with NB = 4 (2 KB per group)
  static_assert(L::kFOff - L::kXOff == L::kXGroups * kXG, "geometry must be sized for 16 rows");
  static_assert(L::kXGroups >= 2 * WN && WN % 2 == 0, "x region must hold two chunks");

  bool any;
  out_col<CH, SWIGLU>(slice, 0, 0, N, &any);

#pragma unroll
  for (int c = 0; c < CH; ++c)
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[c][i][r] = 0.0f;

  const int nst = (nq + 1) >> 1;
  auto issue = [&](int s) {
    const int u = seq + s;
    const int st = u % kRing;
    const uint32_t bar = bar_s + st * 8;
    mbar_expect_tx(bar, L::kStageTx);
    const int row = 4 * (q0 + 2 * s);
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int x = tile_x<CH, SWIGLU>(slice, c, N);
      tma_load_3d(code_s + (st * CH + c) * L::kCodeTile, tq, x, row, z, bar);
      tma_load_3d(scale_s + (st * CH + c) * L::kScaleTile, ts, x, q0 + 2 * s, z, bar);
    }
  };
  if (any && lane == 0) {
    for (int s = 0; s < kRing - 1 && s < nst; ++s) issue(s);
  }

  const int pg = nq <= kXGroups ? ((nq + 1) & ~1) : WN;
  for (int j = warp; j < pg; j += WN) {
    if (j < nq) {
      float v[2][8];
      prep_load_xa(rowptr, M, q0 + j, v);
      prep_store_xa(v, xbuf + j * kXG, &fsc[j]);
    }
  }
  __syncthreads();

  bool ok = true;
  int fail_s = 0;
  const float zq[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  const uint32_t xbuf_s = smem_u32(xbuf) + lane * 16;
  const uint32_t fsc_s = smem_u32(fsc);
  const int h = lane_chunk(g);
  const int hA = lane_chunk(2 * t), hB = lane_chunk(2 * t + 1);
  const int nchunks = (nq + pg - 1) / pg;
  const int sps = pg >> 1;
  for (int pc = 0; pc < nchunks; ++pc) {
    const int buf = pc & 1;
    float nv[2][8];
    const int qn = (pc + 1) * pg + warp;
    const bool more = pc + 1 < nchunks && qn < nq;
    if (more) prep_load_xa(rowptr, M, q0 + qn, nv);
    const int s_end = ((pc + 1) * sps < nst) ? (pc + 1) * sps : nst;
    if (any) {
      for (int s = pc * sps; s < s_end; ++s) {
        if (ok && lane == 0 && s + kRing - 1 < nst) issue(s + kRing - 1);
        const int u = seq + s;
        const int st = u % kRing;
        if (ok) {
          const bool got = mbar_wait(bar_s + st * 8, (u / kRing) & 1, kWaitLimitNs);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            fail_s = s;
            if (lane == 0 && err) atomicCAS(err, 0u, 8u);  // W4A16_ERR_TIMEOUT
          }
        }
        if (ok) {
#pragma unroll (kUnrollGroups)
          for (int j = 0; j < 2; ++j) {
            const int qi = 2 * s + j;
            if (qi < nq) {
              const int r = 4 * j + t;
              const uint32_t coff = r * 128 + ((h ^ (r & 7)) << 4);
              const int xi = buf * pg + (qi - pc * pg);
              const float fg = lds32f(fsc_s + xi * 4);
              const uint32_t xa = xbuf_s + xi * kXG;
              const uint4 A0 = lds128(xa), A1 = lds128(xa + kXChunkBytes);
              const uint4 A2 = lds128(xa + 2 * kXChunkBytes), A3 = lds128(xa + 3 * kXChunkBytes);
              const uint32_t ah0[4] = {A0.x, A0.y, A0.z, A0.w};
              const uint32_t ah1[4] = {A1.x, A1.y, A1.z, A1.w};
              const uint32_t al0[4] = {A2.x, A2.y, A2.z, A2.w};
              const uint32_t al1[4] = {A3.x, A3.y, A3.z, A3.w};
#pragma unroll
              for (int c = 0; c < CH; ++c) {
                const uint4 wq = lds128(code_s + (st * CH + c) * L::kCodeTile + coff);
                const uint32_t srow = scale_s + (st * CH + c) * L::kScaleTile + j * 128;
                const uint4 sa = lds128(srow + hA * 16), sb = lds128(srow + hB * 16);
                const float sA[4] = {__uint_as_float(sa.x) * fg, __uint_as_float(sa.y) * fg,
                                     __uint_as_float(sa.z) * fg, __uint_as_float(sa.w) * fg};
                const float sB[4] = {__uint_as_float(sb.x) * fg, __uint_as_float(sb.y) * fg,
                                     __uint_as_float(sb.z) * fg, __uint_as_float(sb.w) * fg};
                const uint32_t wv[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  uint32_t p[4];
                  unpack_word(wv[i], p);
                  float d[4];
                  mma_f16_zc(d, ah0, p[0], p[1], zq);
                  mma_f16(d, ah1, p[2], p[3]);
                  mma_f16(d, al0, p[0], p[1]);
                  mma_f16(d, al1, p[2], p[3]);
                  acc[c][i][0] = fmaf(sA[i], d[0], acc[c][i][0]);
                  acc[c][i][1] = fmaf(sB[i], d[1], acc[c][i][1]);
                  acc[c][i][2] = fmaf(sA[i], d[2], acc[c][i][2]);
                  acc[c][i][3] = fmaf(sB[i], d[3], acc[c][i][3]);
                }
              }
            }
          }
        }
        __syncwarp();
      }
    }
    if (more)
      prep_store_xa(nv, xbuf + ((buf ^ 1) * pg + warp) * kXG, &fsc[(buf ^ 1) * pg + warp]);
    if (nchunks > 1) __syncthreads();
  }
  if (any && !ok) {
    for (int s = fail_s; s < nst && s < fail_s + kRing; ++s) {
      const int u = seq + s;
      (void)mbar_wait(bar_s + (u % kRing) * 8, (u / kRing) & 1, kWaitLimitNs / 16);
    }
  }
  if (any) seq += nst;
  __syncthreads();
  return ok;
}

// Results of the 9..16-row orientation: for tile c, row half hf (row g + 8 hf) and column
// half e (0: columns 4 h(2t) + i, 1: columns 4 h(2t + 1) + i, i = 0..3) -> 4 values.
template <int CH>
__device__ __forceinline__ float4 xa_result(const float (&acc)[CH][4][4], int c, int hf, int e) {
  const int r = 2 * hf + e;
  return make_float4(acc[c][0][r], acc[c][1][r], acc[c][2][r], acc[c][3][r]);
}

template <int CH, bool SWIGLU>
__device__ __forceinline__ void store_direct_xa(const float (&acc)[CH][4][4], int slice, int N,
                                                int M, float* y) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int hh[2] = {lane_chunk(2 * t), lane_chunk(2 * t + 1)};
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    const int m = g + 8 * hf;
    if (m >= M) continue;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      if (SWIGLU) {
        constexpr int H = CH / 2;
        const int I = N >> 1;
#pragma unroll
        for (int c = 0; c < H; ++c) {
          const int j = 32 * H * slice + 32 * c + 4 * hh[e];
          if (j < I)
            *reinterpret_cast<float4*>(y + (size_t)m * I + j) =
                swiglu4(xa_result<CH>(acc, c, hf, e), xa_result<CH>(acc, c + H, hf, e));
        }
      } else {
#pragma unroll
        for (int c = 0; c < CH; ++c) {
          const int col = 32 * CH * slice + 32 * c + 4 * hh[e];
          if (col < N)
            *reinterpret_cast<float4*>(y + (size_t)m * N + col) = xa_result<CH>(acc, c, hf, e);
        }
      }
    }
  }
}

}  // namespace mma
}  // namespace w4a16
