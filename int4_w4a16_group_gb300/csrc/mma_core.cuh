// Tensor-core weight-streaming core for small M (decode / draft-tree verify).
//
// Each warp owns a slice of 32 weight columns and walks the CTA's K range one group (32 k) at a
// time. Per group it:
//   * receives, through a private cp.async ring in shared memory, one 16-byte chunk per lane of
//     the packed weights (4 consecutive columns of one packed row) and the group's scales;
//   * turns the 4 words into fp16 MMA A-fragments with two bit tricks: (w & 0x000F000F) |
//     0x64006400 is the fp16 pair (1024 + nibble_0, 1024 + nibble_4), and the same mask
//     shifted by 4 gives 1024 + 16 * nibble; one fp16 FMA then yields nibble - 8 exactly;
//   * multiplies them with the activations on the tensor cores (mma.sync m16n8k16, fp16 in,
//     fp32 accumulate) -- the activations enter as two fp16 terms, x * 2^-e = hi + lo with a
//     per-group power-of-two e, which carries 22 significant bits of each float32 activation;
//   * applies the group scale times 2^e to the fresh fp32 group sums with one FMA each.
// The unpacked codes are exact integers, products of codes and fp16 terms are exact in fp32,
// so the only rounding beyond float32 accumulation is the ~2^-22 relative cut of x.
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
// Chunk mapping: lane (g, t) loads columns 4 h(g) .. 4 h(g) + 3 of its slice with
//   h(g) = g / 2 + 4 (g % 2); A tile T (0, 1) uses columns 4 h + 2T (row g) and 4 h + 2T + 1
//   (row g + 8). For the fused SwiGLU slice (16 gate + 16 up columns) even g hold gate
//   columns and odd g the matching up columns, one lane apart by xor 4.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace w4a16 {
namespace mma {

constexpr int kStages = 8;           // cp.async ring depth per warp
constexpr int kStageBytes = 640;     // 512 B of packed words + 128 B of scales
constexpr int kXChunkBytes = 512;    // per (group, n8 block): 32 lanes x 16 B

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
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

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Exact power of two 2^e for e in [-126, 127].
__device__ __forceinline__ float exp2i(int e) { return __int_as_float((e + 127) << 23); }

// One warp prepares the B fragments of one group q (inputs 32q .. 32q + 31) for rows
// 0 .. M-1 (rows >= M are zero): writes NB x 512 B at dst and the group's 2^e at *fscale.
// rowptr(m) returns a pointer to row m of x (float32, 16-byte aligned).
template <int NB, typename RowPtr>
__device__ __forceinline__ void prep_group(const RowPtr& rowptr, int M, int q, char* dst,
                                           float* fscale) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  float v[NB][8];
  float amax = 0.0f;
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
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[b][j]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  // Scale so that the group's largest magnitude lands in [2^14, 2^15): far from fp16
  // overflow (65504) and with the lo term of every element within 2^17 of it still normal.
  int ex = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127;
  if (amax == 0.0f) ex = 0;
  ex = ex < -110 ? -110 : (ex > 110 ? 110 : ex);
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

// Shared-memory layout of one CTA of WN warps with NB n8-blocks:
//   [x fragments: 2 buffers x WN groups x NB x 512 B][2^e per group: 2 x WN floats, padded]
//   [cp.async rings: WN warps x kStages x 640 B]
template <int NB, int WN>
struct Smem {
  static constexpr int kXBytes = 2 * WN * NB * kXChunkBytes;
  static constexpr int kFBytes = ((2 * WN * 4) + 127) / 128 * 128;
  static constexpr int kPipeOff = kXBytes + kFBytes;
  static constexpr int kPipeBytes = WN * kStages * kStageBytes;
  static constexpr int kBytes = kPipeOff + kPipeBytes;
};

// Column of the 4-column chunk lane (g, t) streams in slice `slice`, and whether it exists.
// Plain: the slice is columns 32 slice .. +31.  SwiGLU (N = 2I): the slice is gate columns
// 16 slice .. +15 and up columns I + 16 slice .. +15; even g hold gate, odd g the matching up.
template <bool SWIGLU>
__device__ __forceinline__ void chunk_column(int slice, int g, int N, int* col, bool* valid) {
  if (SWIGLU) {
    const int I = N >> 1;
    const int j = 16 * slice + 4 * (g >> 1);
    *valid = j < I;
    *col = (g & 1) ? I + j : j;
  } else {
    const int h = (g >> 1) + 4 * (g & 1);
    *col = 32 * slice + 4 * h;
    *valid = *col < N;
  }
}

// The CTA's warps stream groups q0 .. q0 + nq - 1 of their slices (slice = slice0 + warp) and
// accumulate, per lane, acc[T][b][r] (A tile T, n8 block b, C register r).
// rowptr(m) -> pointer to row m (< M) of the float32 activations (K floats).
// All threads of the CTA must call this (it synchronizes the CTA between x chunks).
template <int NB, bool SWIGLU, int WN, typename RowPtr>
__device__ __forceinline__ void stream_groups(const RowPtr& rowptr, int M, const int32_t* qw,
                                              const float* sc, int N, int q0, int nq,
                                              int slice0, char* smem, float (&acc)[2][NB][4]) {
  using L = Smem<NB, WN>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  char* xbuf = smem;
  float* fsc = reinterpret_cast<float*>(smem + L::kXBytes);
  char* ring = smem + L::kPipeOff + warp * kStages * kStageBytes;
  const uint32_t ring_s = smem_u32(ring);

  int col;
  bool valid;
  chunk_column<SWIGLU>(slice0 + warp, g, N, &col, &valid);
  const bool warp_active = __any_sync(0xffffffffu, valid);
  const int nbytes = valid ? 16 : 0;
  const int32_t* qsrc = valid ? qw + col : qw;
  const float* ssrc = valid ? sc + col : sc;

#pragma unroll
  for (int T = 0; T < 2; ++T)
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[T][b][r] = 0.0f;

  auto issue = [&](int s) {
    const int q = q0 + s;
    const uint32_t st = ring_s + (s % kStages) * kStageBytes;
    cp_async16(st + lane * 16, qsrc + (size_t)(4 * q + t) * N, nbytes);
    if (t == 0) cp_async16(st + 512 + g * 16, ssrc + (size_t)q * N, nbytes);
  };

  if (warp_active) {
#pragma unroll
    for (int s = 0; s < kStages - 1; ++s) {
      if (s < nq) issue(s);
      cp_async_commit();
    }
  }
  if (warp < nq) prep_group<NB>(rowptr, M, q0 + warp, xbuf + warp * NB * kXChunkBytes, &fsc[warp]);
  __syncthreads();

  const int nchunks = (nq + WN - 1) / WN;
  for (int c = 0; c < nchunks; ++c) {
    const int buf = c & 1;
    const int qn = (c + 1) * WN + warp;
    if (qn < nq)
      prep_group<NB>(rowptr, M, q0 + qn, xbuf + ((buf ^ 1) * WN + warp) * NB * kXChunkBytes,
                     &fsc[(buf ^ 1) * WN + warp]);
    const int iend = (nq - c * WN) < WN ? (nq - c * WN) : WN;
    if (warp_active) {
      for (int i = 0; i < iend; ++i) {
        const int s = c * WN + i;
        if (s + kStages - 1 < nq) issue(s + kStages - 1);
        cp_async_commit();
        cp_async_wait<kStages - 1>();
        __syncwarp();
        const char* st = ring + (s % kStages) * kStageBytes;
        const uint4 wq = *reinterpret_cast<const uint4*>(st + lane * 16);
        const float4 s4 = *reinterpret_cast<const float4*>(st + 512 + g * 16);
        const float fg = fsc[buf * WN + i];
        const char* xb = xbuf + (buf * WN + i) * NB * kXChunkBytes + lane * 16;
        uint4 bf[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) bf[b] = *reinterpret_cast<const uint4*>(xb + b * kXChunkBytes);
        __syncwarp();  // the stage may be refilled by the next issue
        uint32_t p[4][4];
        unpack_word(wq.x, p[0]);
        unpack_word(wq.y, p[1]);
        unpack_word(wq.z, p[2]);
        unpack_word(wq.w, p[3]);
        float d[2][NB][4];
#pragma unroll
        for (int T = 0; T < 2; ++T)
#pragma unroll
          for (int b = 0; b < NB; ++b)
#pragma unroll
            for (int r = 0; r < 4; ++r) d[T][b][r] = 0.0f;
#pragma unroll
        for (int T = 0; T < 2; ++T) {
          const uint32_t a0[4] = {p[2 * T][0], p[2 * T + 1][0], p[2 * T][1], p[2 * T + 1][1]};
          const uint32_t a1[4] = {p[2 * T][2], p[2 * T + 1][2], p[2 * T][3], p[2 * T + 1][3]};
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            mma_f16(d[T][b], a0, bf[b].x, bf[b].y);
            mma_f16(d[T][b], a1, bf[b].z, bf[b].w);
          }
        }
        const float sv[4] = {s4.x * fg, s4.y * fg, s4.z * fg, s4.w * fg};
#pragma unroll
        for (int T = 0; T < 2; ++T)
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            acc[T][b][0] = fmaf(sv[2 * T], d[T][b][0], acc[T][b][0]);
            acc[T][b][1] = fmaf(sv[2 * T], d[T][b][1], acc[T][b][1]);
            acc[T][b][2] = fmaf(sv[2 * T + 1], d[T][b][2], acc[T][b][2]);
            acc[T][b][3] = fmaf(sv[2 * T + 1], d[T][b][3], acc[T][b][3]);
          }
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();
  __syncthreads();  // the ring area may be reused by the caller's epilogue
}

// Per lane: the 4 finished outputs (hi + lo terms) of row m = 4b + t for the lane's chunk.
template <int NB>
__device__ __forceinline__ float4 chunk_result(const float (&acc)[2][NB][4], int b) {
  return make_float4(acc[0][b][0] + acc[0][b][1], acc[0][b][2] + acc[0][b][3],
                     acc[1][b][0] + acc[1][b][1], acc[1][b][2] + acc[1][b][3]);
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

__device__ __forceinline__ float4 shfl_xor4(float4 v, int m) {
  v.x = __shfl_xor_sync(0xffffffffu, v.x, m);
  v.y = __shfl_xor_sync(0xffffffffu, v.y, m);
  v.z = __shfl_xor_sync(0xffffffffu, v.z, m);
  v.w = __shfl_xor_sync(0xffffffffu, v.w, m);
  return v;
}

// Writes the lane's finished outputs straight to y (used when one CTA covers the whole K).
// Plain: y[M, N].  SwiGLU: y[M, N/2] = silu(gate) * up, combined across lane pairs (xor 4).
template <int NB, bool SWIGLU>
__device__ __forceinline__ void store_direct(const float (&acc)[2][NB][4], int slice, int N,
                                             int M, float* y) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  int col;
  bool valid;
  chunk_column<SWIGLU>(slice, g, N, &col, &valid);
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const int m = 4 * b + t;
    float4 v = chunk_result<NB>(acc, b);
    if (SWIGLU) {
      const float4 u = shfl_xor4(v, 4);
      const int I = N >> 1;
      if (!(g & 1) && valid && m < M) {
        float4 o;
        o.x = silu_f(v.x) * u.x;
        o.y = silu_f(v.y) * u.y;
        o.z = silu_f(v.z) * u.z;
        o.w = silu_f(v.w) * u.w;
        *reinterpret_cast<float4*>(y + (size_t)m * I + col) = o;
      }
    } else if (valid && m < M) {
      *reinterpret_cast<float4*>(y + (size_t)m * N + col) = v;
    }
  }
}

}  // namespace mma
}  // namespace w4a16
