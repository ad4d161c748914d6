// Split-K epilogue of the small-M kernels: the CTAs of one thread-block cluster hold partial
// sums of the same output tile over different K ranges and add them through distributed shared
// memory in rank order (deterministic, no global scratch, no atomics).
#pragma once
#include <cuda_bf16.h>

#include "mma_core.cuh"

namespace w4a16 {
namespace mma {

// Output element stores: float32, or bf16 (bit pattern in uint16_t) rounded to nearest even.
__device__ __forceinline__ void store_out(float* y, size_t i, float v) { y[i] = v; }
__device__ __forceinline__ void store_out(uint16_t* y, size_t i, float v) {
  y[i] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
}
// Four consecutive outputs starting at element i of a row of length n: one vector store where
// the four are in the row and aligned, element stores otherwise.
__device__ __forceinline__ void store_out4(float* y, size_t i, int col, int n, float4 v) {
  if (col + 3 < n && (i & 3) == 0) {
    *reinterpret_cast<float4*>(y + i) = v;
    return;
  }
  const float e[4] = {v.x, v.y, v.z, v.w};
  for (int j = 0; j < 4 && col + j < n; ++j) y[i + j] = e[j];
}
__device__ __forceinline__ void store_out4(uint16_t* y, size_t i, int col, int n, float4 v) {
  const float e[4] = {v.x, v.y, v.z, v.w};
  if (col + 3 < n && (i & 3) == 0) {
    uint16_t b[4];
    for (int j = 0; j < 4; ++j) b[j] = __bfloat16_as_ushort(__float2bfloat16_rn(e[j]));
    *reinterpret_cast<uint2*>(y + i) = make_uint2(b[0] | ((uint32_t)b[1] << 16),
                                                  b[2] | ((uint32_t)b[3] << 16));
    return;
  }
  for (int j = 0; j < 4 && col + j < n; ++j) store_out(y, i + j, e[j]);
}
__device__ __forceinline__ void add4(float4& a, const float4& b) {
  a.x += b.x;
  a.y += b.y;
  a.z += b.z;
  a.w += b.w;
}
__device__ __forceinline__ void sts4(uint32_t addr, float4 v) {
  asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"r"(addr), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}
__device__ __forceinline__ float4 lds4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];\n"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
// 16-byte store into the shared memory of another CTA of the cluster; its bytes complete a
// transaction count on that CTA's mbarrier `bar` (both cluster addresses, from mapa_shared).
__device__ __forceinline__ void st_async4(uint32_t addr, float4 v, uint32_t bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, "
      "[%5];\n" ::"r"(addr),
      "r"(__float_as_uint(v.x)), "r"(__float_as_uint(v.y)), "r"(__float_as_uint(v.z)),
      "r"(__float_as_uint(v.w)), "r"(bar)
      : "memory");
}
// The two halves of the hardware cluster barrier (every thread of every CTA of the cluster).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

constexpr int kMaxRanks = 16;  // largest cluster a split over K uses

// Split-K epilogue by pushes. The CK CTAs of a cluster hold partial sums of the same output
// tile (kRows rows, kCols columns; SwiGLU: kCols / 2 gate columns, then the matching up
// columns) over different K ranges. Rank r owns output quads [r per, (r + 1) per) of the tile
// (per = ceil(quads / CK); the last ranks may own fewer or none). Every rank sends each float4
// of its partial tile to the owner of those columns: into its own receive slots with a plain
// store, into a peer's with st.async, whose bytes complete the owner's receive barrier. The
// owner then adds the CK slots of each output in rank order (deterministic, no atomics, no
// global scratch) and writes y (SwiGLU: silu(gate) * up).
// Receive slots, in floats from `buf`: [rank q][row m][half h][P = 4 per owned columns].
template <bool SWIGLU, int kCols, int kRows>
struct SplitKPush {
  static constexpr int kOut = SWIGLU ? kCols / 2 : kCols;  // output columns of the tile
  static_assert(kOut % 4 == 0, "outputs are sent and added four at a time");
  static constexpr int kQuads = kOut / 4;
  static constexpr int kHalves = SWIGLU ? 2 : 1;
  // Receive-slot bytes for any cluster size up to kMaxRanks (CK per <= kQuads + CK - 1).
  static constexpr int kSlotBytes = 4 * kRows * kHalves * (kOut + 4 * (kMaxRanks - 1));

  int CK, rank, per, own;
  uint32_t buf, bar;

  __device__ __forceinline__ SplitKPush(int ck, int r, uint32_t slots, uint32_t recv_bar)
      : CK(ck), rank(r), buf(slots), bar(recv_bar) {
    per = (kQuads + CK - 1) / CK;
    own = max(0, min(per, kQuads - rank * per));
  }
  __device__ __forceinline__ uint32_t slot(int q, int m, int h) const {
    return buf + 16u * (uint32_t)(((q * kRows + m) * kHalves + h) * per);
  }
  // Bytes the peers send this rank for Ms rows.
  __device__ __forceinline__ uint32_t rx_bytes(int Ms) const {
    return (uint32_t)((CK - 1) * Ms * kHalves * own * 16);
  }
  // Sends this rank's partial sums of row m, tile columns lc .. lc + 3 (lc % 4 == 0).
  __device__ __forceinline__ void put(int m, int lc, float4 v) const {
    const int h = (SWIGLU && lc >= kOut) ? 1 : 0;
    const int qd = (lc - h * kOut) >> 2;
    const int r = qd / per;
    const uint32_t a = slot(rank, m, h) + 16u * (uint32_t)(qd - r * per);
    if (r == rank)
      sts4(a, v);
    else
      st_async4(mapa_shared(a, (uint32_t)r), v, mapa_shared(bar, (uint32_t)r));
  }
  // Waits for the peers' bytes (bounded), then adds and stores this rank's outputs of rows
  // [0, Ms) of output tile `tile` of y[., n]. Every thread of the CTA calls it. Returns false if
  // the wait gave up (the outputs are then not written).
  template <typename OutT>
  __device__ __forceinline__ bool finish(int Ms, int tile, int n, OutT* y) const {
    const bool ok = mbar_wait_cluster(bar, 0, kWaitLimitNs);
    // One CTA barrier: this rank's own slots (written by its other threads) are visible, and every
    // thread agrees on the outcome of the wait.
    if (!__syncthreads_and(ok)) return false;
    for (int idx = threadIdx.x; idx < Ms * own; idx += blockDim.x) {
      const int m = idx / own, jq = idx - m * own;
      float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      for (int q = 0; q < CK; ++q) add4(v, lds4(slot(q, m, 0) + 16u * jq));
      if constexpr (SWIGLU) {
        float4 u = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        for (int q = 0; q < CK; ++q) add4(u, lds4(slot(q, m, 1) + 16u * jq));
        v = make_float4(silu_f(v.x) * u.x, silu_f(v.y) * u.y, silu_f(v.z) * u.z,
                        silu_f(v.w) * u.w);
      }
      const int col = tile * kOut + 4 * (rank * per + jq);
      if (col < n) store_out4(y, (size_t)m * n + col, col, n, v);
    }
    return true;
  }
};

}  // namespace mma
}  // namespace w4a16
