// Chained MLP (placeholder until the persistent kernel lands).
#include "internal.h"

namespace coalesce {

uint32_t mlp_max_weight_bytes() { return 160u * 1024u; }

cudaError_t launch_mlp_fused(const DeviceCtx&, int64_t, int, int, int, const void*, const void* const*,
                             const void* const*, void*, int, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace coalesce
