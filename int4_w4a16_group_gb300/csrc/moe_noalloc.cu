// Routed-expert MoE block for callers that cannot allocate device memory.
//
// w4a16_moe_gemm needs a scratch workspace (routing lists, the SwiGLU activations and the
// per-pair outputs) that its caller allocates. Some callers only ever hand over input and output
// buffers: a plugin or foreign-function interface with a fixed signature, or a process whose
// device memory another runtime has already reserved, where a cudaMalloc would fail or stall.
// For them this file keeps one scratch array of fixed size in device memory, created when the
// library's device code is loaded on a GPU and kept by every GPU that loads it until the process
// exits, and runs the ordinary MoE path on it. Nothing here allocates.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/w4a16.h"
#include "internal.h"

namespace {

// The scratch itself. In host code this name is only a stand-in for the device array; the
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_moe_scratch[W4A16_MOE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices];  // device address of g_moe_scratch, per device

// Resolves (once per device, with that device current) the device address of the scratch.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_moe_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" w4a16_status w4a16_moe_gemm_noalloc(const float* x, const int32_t* topk_ids,
                                               const float* topk_w, int T, int topk, int E,
                                               const int32_t* qw_gu, const float* sc_gu,
                                               const int32_t* qw_dn, const float* sc_dn,
                                               float* out, int K, int I, int group,
                                               w4a16_stream_t stream) {
  if (T < 0 || topk <= 0 || E <= 0 || K <= 0 || I <= 0) return W4A16_ERR_ARG;
  // Sizes whose scratch does not fit the fixed array are refused before anything runs.
  if (w4a16_moe_workspace_size(T, topk, E, K, I) > (size_t)W4A16_MOE_STATIC_SCRATCH_BYTES)
    return W4A16_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return W4A16_ERR_CUDA;
  // Every value the MoE path reads from its workspace is written earlier in the same call, so
  // the contents left by a previous call need no clearing.
  return w4a16_moe_gemm(x, topk_ids, topk_w, T, topk, E, qw_gu, sc_gu, qw_dn, sc_dn, out, K, I,
                        group, scratch, (size_t)W4A16_MOE_STATIC_SCRATCH_BYTES, stream);
}
