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

using w4a16::kMaxDevices;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices];  // device address of g_moe_scratch, per device

// Device address of the scratch on the current device. Outside stream capture it is looked up
// on every call (with that device current), so a device reset -- which releases the array and
// loads it again at the next use -- never leaves a stale address behind. Under stream capture
// the address of the last lookup on this device is used, so a captured call needs one earlier
// call on the device outside capture.
cudaError_t scratch_address(cudaStream_t stream, void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(stream, &cs);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (cs == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_moe_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  } else if (!g_scratch_ptr[dev]) {
    return cudaErrorStreamCaptureUnsupported;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" w4a16_status w4a16_moe_gemm_noalloc(const float* x, const int32_t* topk_ids,
                                               const float* topk_w, int T, int topk, int E,
                                               const int32_t* qw_gu, const float* sc_gu,
                                               const int32_t* qw_dn, const float* sc_dn,
                                               float* out, int K, int I, int group,
                                               w4a16_stream_t stream) {
  // The argument checks of w4a16_moe_gemm, in its order, so that both entries answer alike.
  if (group != W4A16_GROUP) return W4A16_ERR_UNSUPPORTED;
  if (T < 0 || topk <= 0 || topk > 64 || E <= 0 || E > 4096) return W4A16_ERR_ARG;
  if (K <= 0 || K % W4A16_GROUP != 0 || I <= 0 || I % W4A16_GROUP != 0) return W4A16_ERR_ARG;
  if (T == 0) return W4A16_OK;
  if (!x || !topk_ids || !topk_w || !qw_gu || !sc_gu || !qw_dn || !sc_dn || !out)
    return W4A16_ERR_ARG;
  if (!aligned16(x) || !aligned16(qw_gu) || !aligned16(sc_gu) || !aligned16(qw_dn) ||
      !aligned16(sc_dn) || !aligned16(out) || !aligned16(topk_ids) || !aligned16(topk_w))
    return W4A16_ERR_ALIGN;
  // Sizes whose scratch does not fit the fixed array are refused before anything runs.
  if (w4a16_moe_workspace_size(T, topk, E, K, I) > (size_t)W4A16_MOE_STATIC_SCRATCH_BYTES)
    return W4A16_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (scratch_address((cudaStream_t)stream, &scratch) != cudaSuccess) return W4A16_ERR_CUDA;
  // Every value the MoE path reads from its workspace is written earlier in the same call, so
  // the contents left by a previous call need no clearing.
  return w4a16_moe_gemm(x, topk_ids, topk_w, T, topk, E, qw_gu, sc_gu, qw_dn, sc_dn, out, K, I,
                        group, scratch, (size_t)W4A16_MOE_STATIC_SCRATCH_BYTES, stream);
}
