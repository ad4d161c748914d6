// PTX helpers shared by the kernels (shared-memory loads, mbarriers, cluster forms, TMA, legacy
// tensor-core MMA) and the fp16 unpack of packed INT4 codes.
//
// Unpack: (w & 0x000F000F) | 0x64006400 is the fp16 pair (1024 + nibble_0, 1024 + nibble_4); the
// mask shifted by 4 gives 1024 + 16 * nibble; one fp16 FMA then yields nibble - 8 exactly. This
// is the magic-number integer-to-float conversion (an integer OR'ed into the mantissa of a power
// of two whose exponent makes the mantissa's last bit worth 1, then the power subtracted), as
// published for INT4/INT8-weight fp16 GEMMs by Kim et al., "Who Says Elephants Can't Run:
// Bringing Large Scale MoE Models into Cloud Scale Production" (2022).
//
// MMA operand mapping (m16n8k16; g = lane / 4, t = lane % 4): A (16 x 16): rows = weight columns,
// k = input index. Lane (g, t) holds the packed word of row 4q + t of group q for two columns
// (A rows g and g + 8). Within the group, MMA k-slot 2t + {0, 1} is input 8t + {0, 4} (k-step
// 0, register a0/a1), slot 2t + 8 + {0, 1} is 8t + {1, 5}; k-step 1 uses 8t + {2, 6} and
// 8t + {3, 7}. Any fixed permutation of k inside a group is allowed because the reduction over
// k does not care about order.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace w4a16 {
namespace mma {

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

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // a barrier wait gives up after 2 s

// Exact power of two 2^e for e in [-126, 127].
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((e + 127) << 23); }

// First 1024-byte aligned address (in the shared window) at or after p.
__device__ __forceinline__ char* align1024(char* p) {
  const uint32_t s = smem_u32(p);
  return p + ((1024u - (s & 1023u)) & 1023u);
}

// 16-byte chunk of a 128-byte tile row that lane group g reads (bank-conflict free with the
// 128-byte swizzle).
__device__ __forceinline__ int lane_chunk(int g) { return (g >> 1) + 4 * (g & 1); }

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

}  // namespace mma
}  // namespace w4a16
