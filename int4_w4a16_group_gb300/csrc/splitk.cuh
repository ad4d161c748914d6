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

template <bool SWIGLU, int kCols, typename OutT = float>
__device__ __forceinline__ void cluster_finish(cg::cluster_group& cluster, float* red, int tile,
                                               int M, int N, OutT* y) {
  constexpr int kOut = kCols / 2;
  const int CK = (int)cluster.dim_blocks().y;
  const int rank = (int)cluster.block_index().y;
  cluster.sync();
  if (SWIGLU) {
    const int I = N >> 1;
    const int per = (kOut + CK - 1) / CK;  // any cluster size: the last ranks may get fewer
    for (int idx = threadIdx.x; idx < M * per; idx += blockDim.x) {
      const int m = idx / per;
      const int o = rank * per + (idx - m * per);
      if (o >= kOut) continue;
      float gs = 0.0f, us = 0.0f;
      for (int q = 0; q < CK; ++q) {
        const float* r = cluster.map_shared_rank(red, q);
        gs += r[m * kCols + o];
        us += r[m * kCols + kOut + o];
      }
      const int out = tile * kOut + o;
      if (out < I) store_out(y, (size_t)m * I + out, silu_f(gs) * us);
    }
  } else {
    const int per = (kCols + CK - 1) / CK;
    for (int idx = threadIdx.x; idx < M * per; idx += blockDim.x) {
      const int m = idx / per;
      const int lc = rank * per + (idx - m * per);
      if (lc >= kCols) continue;
      float s = 0.0f;
      for (int q = 0; q < CK; ++q) s += cluster.map_shared_rank(red, q)[m * kCols + lc];
      const int out = tile * kCols + lc;
      if (out < N) store_out(y, (size_t)m * N + out, s);
    }
  }
  cluster.sync();  // peers may still be reading this CTA's shared memory
}

}  // namespace mma
}  // namespace w4a16
