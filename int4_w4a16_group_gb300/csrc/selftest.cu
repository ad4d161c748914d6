// Self-test of the bounded-wait error path that every streaming and tensor-core kernel uses:
// one thread waits on an mbarrier with the same polled, time-limited wait. Without an arrival
// the phase never completes, the wait gives up after `limit_ns` and the kernel records
// W4A16_ERR_TIMEOUT in the device error word, as a stalled pipeline would, and returns; the
// context stays usable. With `arrive` set the thread arrives first and the wait succeeds.
#include <cuda_runtime.h>

#include "../../include/w4a16.h"
#include "internal.h"
#include "mma_core.cuh"

namespace w4a16 {
namespace {

__global__ void wait_timeout_kernel(int arrive, unsigned long long limit_ns, unsigned int* err) {
  __shared__ __align__(8) unsigned long long bar_storage;
  const uint32_t bar = mma::smem_u32(&bar_storage);
  if (threadIdx.x != 0) return;
  mma::mbar_init(bar, 1);
  mma::mbar_fence_init();
  if (arrive) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
  if (!mma::mbar_wait_poll(bar, 0, limit_ns) && err) atomicCAS(err, 0u, 8u);  // W4A16_ERR_TIMEOUT
}

}  // namespace
}  // namespace w4a16

extern "C" w4a16_status w4a16_selftest_wait(int arrive, int limit_us, w4a16_stream_t stream) {
  if (limit_us < 1 || limit_us > 100000) return W4A16_ERR_ARG;
  unsigned int* err = w4a16::device_error_word();
  if (!err) return W4A16_ERR_CUDA;
  w4a16::wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(
      arrive ? 1 : 0, 1000ull * (unsigned long long)limit_us, err);
  return cudaGetLastError() == cudaSuccess ? W4A16_OK : W4A16_ERR_CUDA;
}
