// Large-M (prefill) bf16 tensor-core path: placeholder until the tcgen05 kernel lands.
#include "internal.h"

namespace w4a16 {

cudaError_t launch_gemm_bf16(const uint16_t*, const int32_t*, const float*, uint16_t*, int, int,
                             int, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace w4a16
