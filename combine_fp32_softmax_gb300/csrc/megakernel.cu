// Forward MegaKernel (placeholder until the persistent task-queue kernel is in).
#include <cuda_runtime.h>

#include "common.cuh"

namespace moe {
int megakernel_fwd(const moe_cfg&, const WsLayout&, uint8_t*, const uint16_t*, const uint16_t*, const uint16_t*,
                   const uint16_t*, const float*, float*, int, cudaStream_t) {
  return MOE_ERR_ARG;
}
}  // namespace moe
