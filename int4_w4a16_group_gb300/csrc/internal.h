// Internal host-side interface between the C-ABI layer (abi.cu) and the kernel translation units.
// Launchers assume their arguments were validated by abi.cu.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

namespace w4a16 {

constexpr int kGroup = 32;

struct DeviceInfo {
  int device;
  int sm_count;
  int cc_major, cc_minor;
  size_t smem_optin;     // largest dynamic shared memory per block
  size_t smem_per_sm;    // shared memory per SM
  size_t smem_reserved;  // shared memory the system reserves per resident block
};
// Properties of the current device (cached per device id).
cudaError_t device_info(DeviceInfo* out);

// Device address of the library's error word (one per device, lazily resolved).
unsigned int* device_error_word();

// Launch data a launcher computes once per device (kernel attributes set, occupancy queried).
// Host threads may race to the first launch: the first one on a device runs `init` under the
// lock and publishes the device's ready bit with release order, so a thread that sees the bit
// (acquire) also sees the finished data.
// Devices 0 .. kMaxDevices - 1 are served (the same bound as the rest of the library); a larger
// id is refused with cudaErrorInvalidDevice.
constexpr int kMaxDevices = 64;

template <typename T>
struct PerDeviceOnce {
  std::atomic<uint64_t> ready{0};
  std::mutex lock;
  T data[kMaxDevices] = {};
  template <typename Init>
  cudaError_t get(int device, Init&& init, const T** out) {
    if (device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
    const int d = device;
    const uint64_t bit = 1ull << d;
    if (!(ready.load(std::memory_order_acquire) & bit)) {
      std::lock_guard<std::mutex> guard(lock);
      if (!(ready.load(std::memory_order_relaxed) & bit)) {
        const cudaError_t e = init(data[d]);
        if (e != cudaSuccess) return e;
        ready.fetch_or(bit, std::memory_order_release);
      }
    }
    *out = &data[d];
    return cudaSuccess;
  }
};

// ---- tmap.cu : TMA descriptor of a row-major [d2][d1][d0] tensor of 4-byte elements, box
// (b0 x b1 x 1); kind 0 = packed codes (int32, 128-byte swizzle), 1 = scales (float32).
cudaError_t make_tmap(CUtensorMap* out, int kind, const void* base, uint64_t d0, uint64_t d1,
                      uint64_t d2, uint32_t b0, uint32_t b1);
// General form: element type, element size and swizzle given explicitly. Out-of-range box
// elements read as zero.
cudaError_t make_tmap_ex(CUtensorMap* out, CUtensorMapDataType dtype, uint32_t elem_bytes,
                         CUtensorMapSwizzle swz, const void* base, uint64_t d0, uint64_t d1,
                         uint64_t d2, uint32_t b0, uint32_t b1);

// Tiled descriptor of 2..5 dimensions: dims[0] contiguous, strides[i] = byte stride of
// dimension i + 1 (any order), box per dimension. Out-of-range box elements read as zero.
cudaError_t make_tmap_nd(CUtensorMap* out, CUtensorMapDataType dtype, CUtensorMapSwizzle swz,
                         const void* base, int rank, const uint64_t* dims,
                         const uint64_t* strides, const uint32_t* box);

// ---- quant.cu
cudaError_t launch_quantize(const float* W, int K, int N, int32_t* qw, float* sc, cudaStream_t s);
cudaError_t launch_dequantize(const int32_t* qw, const float* sc, int K, int N, float* W,
                              cudaStream_t s);

// ---- gemv.cu : small-M weight-streaming kernels.
// Dense: y[M, N] = x[M, K] @ W.  SwiGLU: y[M, N/2] = silu(gate) * up.  Above 16 rows one launch
// covers 16-row slices as grid z, so M <= kGemvMaxRowsPerLaunch per call.
cudaError_t launch_gemv(const float* x, const int32_t* qw, const float* sc, float* y, int M,
                        int N, int K, bool swiglu, cudaStream_t s);
constexpr int kGemvMaxM = 16;

constexpr int kGemvMaxRowsPerLaunch = kGemvMaxM * 4096;
// The same for bf16 activations and bf16 output (y[M, N] = bf16(x @ W)), M <= 16.
cudaError_t launch_gemv_b16(const uint16_t* x, const int32_t* qw, const float* sc, uint16_t* y,
                            int M, int N, int K, cudaStream_t s);


// ---- moe.cu
size_t moe_workspace_size(int T, int topk, int E, int K, int I);
cudaError_t launch_moe(const float* x, const int32_t* ids, const float* w, int T, int topk,
                       int E, const int32_t* qw_gu, const float* sc_gu, const int32_t* qw_dn,
                       const float* sc_dn, float* out, int K, int I, void* ws, size_t ws_bytes,
                       cudaStream_t s);
size_t moe_block_workspace_size(int T, int topk, int E, int K, int I, int Is);
cudaError_t launch_moe_block(const float* x, const int32_t* ids, const float* w, int T, int topk,
                             int E, const int32_t* qw_gu, const float* sc_gu,
                             const int32_t* qw_dn, const float* sc_dn, const int32_t* qs_gu,
                             const float* ss_gu, const int32_t* qs_dn, const float* ss_dn, int Is,
                             float* out, int K, int I, void* ws, size_t ws_bytes,
                             cudaStream_t s);
cudaError_t launch_topk_softmax(const float* logits, float* weights, int T, int topk,
                                cudaStream_t s);

// ---- prefill.cu : tcgen05 path
cudaError_t launch_gemm_bf16(const uint16_t* x, const int32_t* qw, const float* sc, uint16_t* y,
                             int M, int N, int K, cudaStream_t s);

}  // namespace w4a16
