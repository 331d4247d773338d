// q4k_gemm.cu -- prefill projection (placeholder until the tcgen05 kernel lands).
#include "q4k_device.cuh"
#include "q4k_internal.h"

namespace q4k {
cudaError_t launch_gemm(const void *, int64_t, int64_t, const void *, int64_t, int64_t, void *,
                        int64_t, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace q4k
