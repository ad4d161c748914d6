// CUDA-core building blocks shared by the dense and the grouped (MoE) weight-streaming kernels.
//
// A CTA of 8 warps owns a tile of 128 output columns; each lane owns 4 adjacent columns and
// reads them with one 16-byte load per packed row (8 k). Warps split the CTA's K range by
// groups of 32 k; per group the lane forms the exact code values, accumulates sum_k x[m,k]*q
// for the group, then applies the group scale with one FMA per (row, column) -- the scale is
// fused into the reduction, one multiply per 32 k.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace w4a16 {
namespace simt {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTileN = 128;  // output columns per CTA tile (SwiGLU: 64 gate + 64 up)

// Exact float value of (nibble j of w) - 8: placing a 4-bit integer v in the low mantissa bits
// of 2^23 gives the float 2^23 + v exactly; subtracting 2^23 + 8 is exact too.
__device__ __forceinline__ float code_value(uint32_t w, int j) {
  return __uint_as_float(0x4B000000u | ((w >> (4 * j)) & 0xFu)) - 8388616.0f;
}

__device__ __forceinline__ float f4_get(const float4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// Column layout of a tile. Plain: lane l owns columns 128*tile + 4l .. +3.
// SwiGLU (gate | up halves of width I): lanes 0..15 own gate columns 64*tile + 4l .. +3,
// lanes 16..31 the matching up columns I + 64*tile + 4(l-16) .. +3.
template <bool SWIGLU>
__device__ __forceinline__ void lane_columns(int tile, int lane, int N, int* col, bool* valid) {
  if (SWIGLU) {
    const int I = N >> 1;
    const int j = 64 * tile + 4 * (lane & 15);
    *valid = j < I;
    *col = (lane < 16) ? j : I + j;
  } else {
    *col = kTileN * tile + 4 * lane;
    *valid = *col < N;
  }
}

// Accumulates, for this lane's 4 columns and MM rows, sum over groups g = g_begin, g_begin +
// g_step, ... < g_end of s[g, c] * sum_{k in g} x[m, k] * q[k, c] into acc.
// xrow[m] points at row m of the activations (K floats, 16-byte aligned).
template <int MM>
__device__ __forceinline__ void accumulate_groups(const float* const* xrow, const int32_t* qw,
                                                  const float* sc, int N, int col, int g_begin,
                                                  int g_end, int g_step, float (&acc)[MM][4]) {
  const size_t rstride = (size_t)(N >> 2);  // int4 units per packed row
  const int4* qp = reinterpret_cast<const int4*>(qw + col);
  const float4* sp = reinterpret_cast<const float4*>(sc + col);
  for (int g = g_begin; g < g_end; g += g_step) {
    int4 wq[4];
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) wq[kb] = __ldg(qp + (size_t)(4 * g + kb) * rstride);
    const float4 s4 = __ldg(sp + (size_t)g * rstride);
    float part[MM][4];
#pragma unroll
    for (int m = 0; m < MM; ++m)
#pragma unroll
      for (int c = 0; c < 4; ++c) part[m][c] = 0.0f;
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) {
      const uint32_t wv[4] = {(uint32_t)wq[kb].x, (uint32_t)wq[kb].y, (uint32_t)wq[kb].z,
                              (uint32_t)wq[kb].w};
#pragma unroll
      for (int jq = 0; jq < 2; ++jq) {
        float4 xv[MM];
#pragma unroll
        for (int m = 0; m < MM; ++m)
          xv[m] = __ldg(reinterpret_cast<const float4*>(xrow[m] + 32 * g + 8 * kb + 4 * jq));
#pragma unroll
        for (int c = 0; c < 4; ++c) {
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const float v = code_value(wv[c], 4 * jq + jj);
#pragma unroll
            for (int m = 0; m < MM; ++m) part[m][c] = fmaf(f4_get(xv[m], jj), v, part[m][c]);
          }
        }
      }
    }
    const float s[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
    for (int m = 0; m < MM; ++m)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[m][c] = fmaf(s[c], part[m][c], acc[m][c]);
  }
}

// Writes each warp's partial sums to red[warp][m][slot] and sums the warps, in warp order,
// into red[0][m][slot]. Ends with the CTA synchronized.
template <int MM>
__device__ __forceinline__ void reduce_warps(float* red, const float (&acc)[MM][4], int warp,
                                             int lane) {
#pragma unroll
  for (int m = 0; m < MM; ++m)
    *reinterpret_cast<float4*>(&red[(warp * MM + m) * kTileN + 4 * lane]) =
        make_float4(acc[m][0], acc[m][1], acc[m][2], acc[m][3]);
  __syncthreads();
  for (int idx = threadIdx.x; idx < MM * kTileN; idx += kThreads) {
    float s = red[idx];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) s += red[w * MM * kTileN + idx];
    red[idx] = s;
  }
  __syncthreads();
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

}  // namespace simt
}  // namespace w4a16
