// q4k_moe.cu -- routed-expert decode FFN (placeholder until the kernel lands).
#include "q4k_device.cuh"
#include "q4k_internal.h"

namespace q4k {
size_t moe_workspace_size(int32_t, int32_t, int32_t, int64_t, int64_t) { return 16; }
cudaError_t launch_moe(const void *, const void *, const void *, int64_t, int32_t, int64_t, int64_t,
                       const void *, int32_t, int64_t, const int32_t *, const float *, int32_t,
                       float *, int64_t, void *, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace q4k
