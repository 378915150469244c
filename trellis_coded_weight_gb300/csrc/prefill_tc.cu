// prefill_tc.cu -- placeholder until the tcgen05 prefill GEMM lands.
#include <cuda_runtime.h>
#include "launch.h"
namespace trellis {
cudaError_t launch_gemm_prefill(const uint32_t*, const uint16_t*, const uint16_t*, uint16_t*, int, int, int,
                                int64_t, int64_t, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace trellis
