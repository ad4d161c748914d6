// C ABI of libw4a16.so (declared in include/w4a16.h): argument checks, dispatch to the kernel
// launchers, the raw .qw/.sc loader and the name -> weight registry behind linear().
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <map>
#include <mutex>
#include <string>

#include "../../include/w4a16.h"
#include "internal.h"

#ifndef W4A16_B16_STREAM_MAX_M
#define W4A16_B16_STREAM_MAX_M 16
#endif

namespace w4a16 {

namespace {
thread_local int g_last_cuda_error = 0;

DeviceInfo g_info[kMaxDevices];
bool g_info_valid[kMaxDevices];
std::mutex g_info_mutex;

// Error word written by kernels that give up a bounded wait (one copy per device).
__device__ unsigned int g_device_error;
unsigned int* g_error_ptr[kMaxDevices];
}  // namespace

cudaError_t device_info(DeviceInfo* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_info_mutex);
  if (!g_info_valid[dev]) {
    DeviceInfo d;
    d.device = dev;
    int v = 0;
    if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return e;
    d.sm_count = v;
    if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return e;
    d.cc_major = v;
    if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return e;
    d.cc_minor = v;
    if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) !=
        cudaSuccess)
      return e;
    d.smem_optin = (size_t)v;
    if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
        cudaSuccess)
      return e;
    d.smem_per_sm = (size_t)v;
    if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrReservedSharedMemoryPerBlock, dev)) !=
        cudaSuccess)
      return e;
    d.smem_reserved = (size_t)v;
    g_info[dev] = d;
    g_info_valid[dev] = true;
  }
  *out = g_info[dev];
  return cudaSuccess;
}

unsigned int* device_error_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_info_mutex);
  if (!g_error_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    g_error_ptr[dev] = static_cast<unsigned int*>(p);
  }
  return g_error_ptr[dev];
}

}  // namespace w4a16

using namespace w4a16;

namespace {

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

inline w4a16_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return W4A16_OK;
  g_last_cuda_error = (int)e;
  return W4A16_ERR_CUDA;
}

// Common checks of a weight matrix description.
inline w4a16_status check_weights(const int32_t* qw, const float* sc, int K, int N, int group) {
  if (group != W4A16_GROUP) return W4A16_ERR_UNSUPPORTED;
  if (K <= 0 || K % W4A16_GROUP != 0 || N < 0 || N % 4 != 0) return W4A16_ERR_ARG;
  if (N > 0 && (!qw || !sc)) return W4A16_ERR_ARG;
  if (!aligned16(qw) || !aligned16(sc)) return W4A16_ERR_ALIGN;
  return W4A16_OK;
}

w4a16_status gemm_impl(const float* x, const int32_t* qw, const float* sc, float* y, int M,
                       int N, int K, int group, bool swiglu, cudaStream_t stream) {
  w4a16_status st = check_weights(qw, sc, K, N, group);
  if (st != W4A16_OK) return st;
  if (M < 0) return W4A16_ERR_ARG;
  if (swiglu && N % 8 != 0) return W4A16_ERR_ARG;
  if (M == 0 || N == 0) return W4A16_OK;
  if (!x || !y) return W4A16_ERR_ARG;
  if (!aligned16(x) || !aligned16(y)) return W4A16_ERR_ALIGN;
  const int n_out = swiglu ? N / 2 : N;
  for (int r = 0; r < M; r += kGemvMaxRowsPerLaunch) {
    const int rows = (M - r) < kGemvMaxRowsPerLaunch ? (M - r) : kGemvMaxRowsPerLaunch;
    cudaError_t e = launch_gemv(x + (size_t)r * K, qw, sc, y + (size_t)r * n_out, rows, N, K,
                                swiglu, stream);
    if (e != cudaSuccess) return cuda_status(e);
  }
  return W4A16_OK;
}

}  // namespace

struct w4a16_registry {
  struct Entry {
    const int32_t* qw;
    const float* sc;
    int K, N;
  };
  std::map<std::string, Entry> map;
  mutable std::mutex mu;
};

extern "C" {

const char* w4a16_status_string(w4a16_status s) {
  switch (s) {
    case W4A16_OK: return "W4A16_OK";
    case W4A16_ERR_ARG: return "W4A16_ERR_ARG: invalid size or pointer argument";
    case W4A16_ERR_ALIGN: return "W4A16_ERR_ALIGN: tensor pointer not 16-byte aligned";
    case W4A16_ERR_UNSUPPORTED: return "W4A16_ERR_UNSUPPORTED: unsupported configuration";
    case W4A16_ERR_WORKSPACE: return "W4A16_ERR_WORKSPACE: workspace missing or too small";
    case W4A16_ERR_CUDA: return "W4A16_ERR_CUDA: CUDA call or kernel launch failed";
    case W4A16_ERR_NOT_FOUND: return "W4A16_ERR_NOT_FOUND: no quantized weight under that name";
    case W4A16_ERR_IO: return "W4A16_ERR_IO: file missing, unreadable or of the wrong size";
    case W4A16_ERR_TIMEOUT: return "W4A16_ERR_TIMEOUT: a kernel gave up a bounded wait";
  }
  return "W4A16_ERR_?: unknown status";
}

int w4a16_abi_version(void) { return W4A16_ABI_VERSION; }

int w4a16_last_cuda_error(void) { return g_last_cuda_error; }

w4a16_status w4a16_quantize(const float* W, int K, int N, int group, int32_t* qw, float* sc,
                            w4a16_stream_t stream) {
  w4a16_status st = check_weights(qw, sc, K, N, group);
  if (st != W4A16_OK) return st;
  if (N == 0) return W4A16_OK;
  if (!W) return W4A16_ERR_ARG;
  if (!aligned16(W)) return W4A16_ERR_ALIGN;
  return cuda_status(launch_quantize(W, K, N, qw, sc, (cudaStream_t)stream));
}

w4a16_status w4a16_dequantize(const int32_t* qw, const float* sc, int K, int N, int group,
                              float* W, w4a16_stream_t stream) {
  w4a16_status st = check_weights(qw, sc, K, N, group);
  if (st != W4A16_OK) return st;
  if (N == 0) return W4A16_OK;
  if (!W) return W4A16_ERR_ARG;
  if (!aligned16(W)) return W4A16_ERR_ALIGN;
  return cuda_status(launch_dequantize(qw, sc, K, N, W, (cudaStream_t)stream));
}

w4a16_status w4a16_gemm(const float* x, const int32_t* qw, const float* sc, float* y, int M,
                        int N, int K, int group, w4a16_stream_t stream) {
  return gemm_impl(x, qw, sc, y, M, N, K, group, false, (cudaStream_t)stream);
}

w4a16_status w4a16_gemm_swiglu(const float* x, const int32_t* qw_gu, const float* sc_gu,
                               float* y, int M, int N2, int K, int group,
                               w4a16_stream_t stream) {
  return gemm_impl(x, qw_gu, sc_gu, y, M, N2, K, group, true, (cudaStream_t)stream);
}

w4a16_status w4a16_gemm_bf16(const uint16_t* x, const int32_t* qw, const float* sc, uint16_t* y,
                             int M, int N, int K, int group, w4a16_stream_t stream) {
  w4a16_status st = check_weights(qw, sc, K, N, group);
  if (st != W4A16_OK) return st;
  if (M < 0 || K % 64 != 0 || N % 8 != 0) return W4A16_ERR_ARG;
  if (M == 0 || N == 0) return W4A16_OK;
  if (!x || !y) return W4A16_ERR_ARG;
  if (!aligned16(x) || !aligned16(y)) return W4A16_ERR_ALIGN;
  DeviceInfo di;
  cudaError_t e = device_info(&di);
  if (e != cudaSuccess) return cuda_status(e);
  if (di.cc_major != 10 || di.cc_minor != 3) return W4A16_ERR_UNSUPPORTED;
  // Up to W4A16_B16_STREAM_MAX_M rows the op is weight streaming (the small-M kernels in bf16
  // form, 16-row slices); larger M is the tensor-core contraction.
  if (M <= W4A16_B16_STREAM_MAX_M) {
    for (int m0 = 0; m0 < M && e == cudaSuccess; m0 += kGemvMaxM) {
      const int mc = M - m0 < kGemvMaxM ? M - m0 : kGemvMaxM;
      e = launch_gemv_b16(x + (size_t)m0 * K, qw, sc, y + (size_t)m0 * N, mc, N, K,
                          (cudaStream_t)stream);
    }
  } else {
    e = launch_gemm_bf16(x, qw, sc, y, M, N, K, (cudaStream_t)stream);
  }
  if (e == cudaErrorNotSupported) return W4A16_ERR_UNSUPPORTED;
  return cuda_status(e);
}

size_t w4a16_moe_workspace_size(int T, int topk, int E, int K, int I) {
  if (T < 0 || topk <= 0 || E <= 0 || K <= 0 || I <= 0) return 0;
  return moe_workspace_size(T, topk, E, K, I);
}

w4a16_status w4a16_moe_gemm(const float* x, const int32_t* topk_ids, const float* topk_w, int T,
                            int topk, int E, const int32_t* qw_gu, const float* sc_gu,
                            const int32_t* qw_dn, const float* sc_dn, float* out, int K, int I,
                            int group, void* workspace, size_t ws_bytes,
                            w4a16_stream_t stream) {
  if (group != W4A16_GROUP) return W4A16_ERR_UNSUPPORTED;
  if (T < 0 || topk <= 0 || topk > 64 || E <= 0 || E > 4096) return W4A16_ERR_ARG;
  if (K <= 0 || K % W4A16_GROUP != 0 || I <= 0 || I % W4A16_GROUP != 0) return W4A16_ERR_ARG;
  if (T == 0) return W4A16_OK;
  if (!x || !topk_ids || !topk_w || !qw_gu || !sc_gu || !qw_dn || !sc_dn || !out)
    return W4A16_ERR_ARG;
  if (!aligned16(x) || !aligned16(qw_gu) || !aligned16(sc_gu) || !aligned16(qw_dn) ||
      !aligned16(sc_dn) || !aligned16(out) || !aligned16(topk_ids) || !aligned16(topk_w))
    return W4A16_ERR_ALIGN;
  const size_t need = moe_workspace_size(T, topk, E, K, I);
  if (!workspace || ws_bytes < need) return W4A16_ERR_WORKSPACE;
  if (!aligned16(workspace)) return W4A16_ERR_ALIGN;
  return cuda_status(launch_moe(x, topk_ids, topk_w, T, topk, E, qw_gu, sc_gu, qw_dn, sc_dn, out,
                                K, I, workspace, ws_bytes, (cudaStream_t)stream));
}

size_t w4a16_moe_block_workspace_size(int T, int topk, int E, int K, int I, int Is) {
  if (T < 0 || topk <= 0 || E <= 0 || K <= 0 || I <= 0 || Is <= 0) return 0;
  return moe_block_workspace_size(T, topk, E, K, I, Is);
}

w4a16_status w4a16_moe_block(const float* x, const int32_t* topk_ids, const float* topk_w, int T,
                             int topk, int E, const int32_t* qw_gu, const float* sc_gu,
                             const int32_t* qw_dn, const float* sc_dn, const int32_t* qs_gu,
                             const float* ss_gu, const int32_t* qs_dn, const float* ss_dn, int Is,
                             float* out, int K, int I, int group, void* workspace,
                             size_t ws_bytes, w4a16_stream_t stream) {
  if (group != W4A16_GROUP) return W4A16_ERR_UNSUPPORTED;
  if (T < 0 || topk <= 0 || topk > 64 || E <= 0 || E > 4096) return W4A16_ERR_ARG;
  if (K <= 0 || K % W4A16_GROUP != 0 || I <= 0 || I % W4A16_GROUP != 0 || Is <= 0 ||
      Is % W4A16_GROUP != 0)
    return W4A16_ERR_ARG;
  if (T == 0) return W4A16_OK;
  if (!x || !topk_ids || !topk_w || !qw_gu || !sc_gu || !qw_dn || !sc_dn || !qs_gu || !ss_gu ||
      !qs_dn || !ss_dn || !out)
    return W4A16_ERR_ARG;
  if (!aligned16(x) || !aligned16(qw_gu) || !aligned16(sc_gu) || !aligned16(qw_dn) ||
      !aligned16(sc_dn) || !aligned16(qs_gu) || !aligned16(ss_gu) || !aligned16(qs_dn) ||
      !aligned16(ss_dn) || !aligned16(out) || !aligned16(topk_ids) || !aligned16(topk_w))
    return W4A16_ERR_ALIGN;
  const size_t need = moe_block_workspace_size(T, topk, E, K, I, Is);
  if (!workspace || ws_bytes < need) return W4A16_ERR_WORKSPACE;
  if (!aligned16(workspace)) return W4A16_ERR_ALIGN;
  return cuda_status(launch_moe_block(x, topk_ids, topk_w, T, topk, E, qw_gu, sc_gu, qw_dn, sc_dn,
                                      qs_gu, ss_gu, qs_dn, ss_dn, Is, out, K, I, workspace,
                                      ws_bytes, (cudaStream_t)stream));
}

w4a16_status w4a16_topk_softmax(const float* logits, float* weights, int T, int topk,
                                w4a16_stream_t stream) {
  if (T < 0 || topk <= 0 || topk > 32) return W4A16_ERR_ARG;
  if (T == 0) return W4A16_OK;
  if (!logits || !weights) return W4A16_ERR_ARG;
  if (!aligned16(logits) || !aligned16(weights)) return W4A16_ERR_ALIGN;
  return cuda_status(launch_topk_softmax(logits, weights, T, topk, (cudaStream_t)stream));
}

w4a16_status w4a16_load_qw_sc(const char* qw_path, const char* sc_path, int K, int N, int group,
                              int32_t* qw, float* sc) {
  w4a16_status st = check_weights(qw, sc, K, N, group);
  if (st != W4A16_OK) return st;
  if (!qw_path || !sc_path) return W4A16_ERR_ARG;
  const size_t qbytes = (size_t)(K / 8) * N * sizeof(int32_t);
  const size_t sbytes = (size_t)(K / W4A16_GROUP) * N * sizeof(float);
  const char* paths[2] = {qw_path, sc_path};
  const size_t sizes[2] = {qbytes, sbytes};
  void* dsts[2] = {qw, sc};
  // Check both files before copying anything.
  for (int f = 0; f < 2; ++f) {
    FILE* fp = fopen(paths[f], "rb");
    if (!fp) return W4A16_ERR_IO;
    const bool seek_ok = fseek(fp, 0, SEEK_END) == 0;
    const long len = seek_ok ? ftell(fp) : -1;
    fclose(fp);
    if (len < 0 || (size_t)len != sizes[f]) return W4A16_ERR_IO;
  }
  for (int f = 0; f < 2; ++f) {
    if (sizes[f] == 0) continue;
    FILE* fp = fopen(paths[f], "rb");
    if (!fp) return W4A16_ERR_IO;
    void* host = malloc(sizes[f]);
    if (!host) {
      fclose(fp);
      return W4A16_ERR_IO;
    }
    const size_t got = fread(host, 1, sizes[f], fp);
    fclose(fp);
    if (got != sizes[f]) {
      free(host);
      return W4A16_ERR_IO;
    }
    cudaError_t e = cudaMemcpy(dsts[f], host, sizes[f], cudaMemcpyHostToDevice);
    free(host);
    if (e != cudaSuccess) return cuda_status(e);
  }
  return W4A16_OK;
}

w4a16_registry* w4a16_registry_create(void) { return new (std::nothrow) w4a16_registry(); }

void w4a16_registry_destroy(w4a16_registry* reg) { delete reg; }

w4a16_status w4a16_registry_add(w4a16_registry* reg, const char* name, const int32_t* qw,
                                const float* sc, int K, int N, int group) {
  if (!reg || !name || !name[0]) return W4A16_ERR_ARG;
  w4a16_status st = check_weights(qw, sc, K, N, group);
  if (st != W4A16_OK) return st;
  std::lock_guard<std::mutex> lock(reg->mu);
  reg->map[name] = w4a16_registry::Entry{qw, sc, K, N};
  return W4A16_OK;
}

w4a16_status w4a16_registry_find(const w4a16_registry* reg, const char* name, int* K, int* N) {
  if (!reg || !name) return W4A16_ERR_ARG;
  std::lock_guard<std::mutex> lock(reg->mu);
  auto it = reg->map.find(name);
  if (it == reg->map.end()) return W4A16_ERR_NOT_FOUND;
  if (K) *K = it->second.K;
  if (N) *N = it->second.N;
  return W4A16_OK;
}

static w4a16_status linear_impl(const w4a16_registry* reg, const char* name, const float* x,
                                float* y, int M, bool swiglu, w4a16_stream_t stream) {
  if (!reg || !name) return W4A16_ERR_ARG;
  w4a16_registry::Entry e;
  {
    std::lock_guard<std::mutex> lock(reg->mu);
    auto it = reg->map.find(name);
    if (it == reg->map.end()) return W4A16_ERR_NOT_FOUND;  // no silent float fallback
    e = it->second;
  }
  return gemm_impl(x, e.qw, e.sc, y, M, e.N, e.K, W4A16_GROUP, swiglu, (cudaStream_t)stream);
}

w4a16_status w4a16_linear(const w4a16_registry* reg, const char* name, const float* x, float* y,
                          int M, w4a16_stream_t stream) {
  return linear_impl(reg, name, x, y, M, false, stream);
}

w4a16_status w4a16_linear_swiglu(const w4a16_registry* reg, const char* name, const float* x,
                                 float* y, int M, w4a16_stream_t stream) {
  return linear_impl(reg, name, x, y, M, true, stream);
}

w4a16_status w4a16_device_error(int* code) {
  if (!code) return W4A16_ERR_ARG;
  unsigned int* p = device_error_word();
  if (!p) return cuda_status(cudaGetLastError());
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_status(e);
  unsigned int v = 0;
  e = cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_status(e);
  const unsigned int zero = 0;
  e = cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_status(e);
  *code = (int)v;
  return W4A16_OK;
}

}  // extern "C"
