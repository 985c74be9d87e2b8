// Placeholder until the tcgen05 attention kernel lands: reports "not supported".
#include "common.cuh"

namespace sage {
cudaError_t launch_attention_tc(const Bundle&, int64_t, int64_t, int64_t, float, const Out&, int*, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace sage
