// Quantize + pack, and unpack + dequantize, of the INT4 group-32 weight format.
//
// Format (page "The Weight of Precision: Building Native INT4 Quantization for a Custom
// Speculative Decoding Engine", section "The Kernel: w4a16_gemm"): symmetric codes,
// value = nibble - 8, eight nibbles per int32 along K, one float32 scale per 32 rows of K per
// output column. Scale rule absmax/7 and half-to-even rounding of the float32 quotient are the
// readings this library documents in w4a16.h.
#include "internal.h"

namespace w4a16 {
namespace {

// One thread per (group g, column n): 32 strided loads (coalesced across the warp along n),
// one scale, four packed words.
__global__ void quantize_kernel(const float* __restrict__ W, int K, int N,
                                int32_t* __restrict__ qw, float* __restrict__ sc) {
  const long long total = (long long)(K / kGroup) * N;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int g = (int)(idx / N);
    const int n = (int)(idx - (long long)g * N);
    const float* col = W + (size_t)g * kGroup * N + n;
    float v[kGroup];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < kGroup; ++i) {
      v[i] = __ldg(col + (size_t)i * N);
      amax = fmaxf(amax, fabsf(v[i]));
    }
    const float s = __fdiv_rn(amax, 7.0f);  // IEEE float32 quotient
    sc[(size_t)g * N + n] = s;
#pragma unroll
    for (int w = 0; w < kGroup / 8; ++w) {
      uint32_t word = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float r = 0.0f;
        if (s != 0.0f) r = rintf(__fdiv_rn(v[8 * w + j], s));  // half to even
        r = fminf(fmaxf(r, -8.0f), 7.0f);
        word |= (uint32_t)((int)r + 8) << (4 * j);
      }
      qw[(size_t)(4 * g + w) * N + n] = (int32_t)word;
    }
  }
}

// One thread per (word row i, column n): eight codes times the group scale, rounded to float32.
__global__ void dequantize_kernel(const int32_t* __restrict__ qw, const float* __restrict__ sc,
                                  int K, int N, float* __restrict__ W) {
  const long long total = (long long)(K / 8) * N;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int i = (int)(idx / N);
    const int n = (int)(idx - (long long)i * N);
    const uint32_t word = (uint32_t)__ldg(qw + idx);
    const float s = __ldg(sc + (size_t)(i / 4) * N + n);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int q = (int)((word >> (4 * j)) & 0xFu) - 8;
      W[(size_t)(8 * i + j) * N + n] = (float)q * s;
    }
  }
}

// Grid-stride launch size: one CTA per `block` items, at most 64 CTAs per SM of this device.
cudaError_t grid_for(long long total, int block, int* grid) {
  DeviceInfo di;
  const cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return e;
  long long b = (total + block - 1) / block;
  const long long cap = (long long)di.sm_count * 64;
  if (b > cap) b = cap;
  *grid = (int)(b < 1 ? 1 : b);
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_quantize(const float* W, int K, int N, int32_t* qw, float* sc, cudaStream_t s) {
  const long long total = (long long)(K / kGroup) * N;
  int grid = 0;
  const cudaError_t e = grid_for(total, 256, &grid);
  if (e != cudaSuccess) return e;
  quantize_kernel<<<grid, 256, 0, s>>>(W, K, N, qw, sc);
  return cudaGetLastError();
}

cudaError_t launch_dequantize(const int32_t* qw, const float* sc, int K, int N, float* W,
                              cudaStream_t s) {
  const long long total = (long long)(K / 8) * N;
  int grid = 0;
  const cudaError_t e = grid_for(total, 256, &grid);
  if (e != cudaSuccess) return e;
  dequantize_kernel<<<grid, 256, 0, s>>>(qw, sc, K, N, W);
  return cudaGetLastError();
}

}  // namespace w4a16
