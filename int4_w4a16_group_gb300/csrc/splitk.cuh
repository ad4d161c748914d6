// Split-K epilogue of the small-M kernels: the CTAs of one thread-block cluster hold partial
// sums of the same output tile over different K ranges and add them through distributed shared
// memory in rank order (deterministic, no global scratch, no atomics).
#pragma once
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "mma_core.cuh"

namespace w4a16 {
namespace mma {

namespace cg = cooperative_groups;

// Every CTA of the cluster has written its partial tile red[M rows][kCols] (SwiGLU: kOut gate
// sums, then the kOut matching up sums); rank r finishes its share of the columns over all
// ranks in rank order and writes y (SwiGLU: silu(gate) * up).
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
// 16-byte load from the shared memory of a CTA of the cluster (address from mapa_shared).
__device__ __forceinline__ float4 ld_cluster4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];\n"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ void add4(float4& a, const float4& b) {
  a.x += b.x;
  a.y += b.y;
  a.z += b.z;
  a.w += b.w;
}
// Sum over the cluster's ranks, in rank order, of the float4 at shared address `addr` (the same
// offset in every CTA). All loads of a batch are issued before the adds.
__device__ __forceinline__ float4 rank_sum4(uint32_t addr, int CK) {
  float4 s = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  for (int q0 = 0; q0 < CK; q0 += 4) {
    float4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (q0 + j < CK) v[j] = ld_cluster4(mapa_shared(addr, (uint32_t)(q0 + j)));
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (q0 + j < CK) add4(s, v[j]);
  }
  return s;
}

template <bool SWIGLU, int kCols, typename OutT = float>
__device__ __forceinline__ void cluster_finish(cg::cluster_group& cluster, float* red, int tile,
                                               int M, int N, OutT* y) {
  constexpr int kOut = SWIGLU ? kCols / 2 : kCols;  // output columns of the tile
  static_assert(kOut % 4 == 0, "the tile's outputs are reduced four at a time");
  constexpr int kQuads = kOut / 4;
  const int CK = (int)cluster.dim_blocks().y;
  const int rank = (int)cluster.block_index().y;
  const int per = (kQuads + CK - 1) / CK;  // any cluster size: the last ranks may get fewer
  const int n = SWIGLU ? N >> 1 : N;
  const uint32_t red_s = (uint32_t)__cvta_generic_to_shared(red);
  cluster.sync();  // every rank's partial tile is written
  for (int idx = threadIdx.x; idx < M * per; idx += blockDim.x) {
    const int m = idx / per;
    const int qd = rank * per + (idx - m * per);
    if (qd >= kQuads) continue;
    const int o = 4 * qd;
    const uint32_t a = red_s + 4u * (uint32_t)(m * kCols + o);
    float4 v = rank_sum4(a, CK);
    if constexpr (SWIGLU) {
      const float4 u = rank_sum4(a + 4u * kOut, CK);
      v = make_float4(silu_f(v.x) * u.x, silu_f(v.y) * u.y, silu_f(v.z) * u.z, silu_f(v.w) * u.w);
    }
    const int col = tile * kOut + o;
    if (col < n) store_out4(y, (size_t)m * n + col, col, n, v);
  }
  // Peers may still be reading this CTA's shared memory: it stays until every rank is done.
  asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

}  // namespace mma
}  // namespace w4a16
