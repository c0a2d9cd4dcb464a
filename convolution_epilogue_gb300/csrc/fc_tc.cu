// fc_tc.cu -- tcgen05 tensor-core path (placeholder until the kernel lands).
#include "fc_internal.h"

namespace fc {
bool tc_supported(const ConvProblem &, int) { return false; }
cudaError_t tc_launch(const ConvProblem &, int, void *, const WsLayout &,
                      cudaStream_t, int *) {
  return cudaErrorNotSupported;
}
int tc_pool_tiles_per_image(const ConvProblem &) { return 0; }
size_t tc_weight_bytes(const ConvProblem &) { return 0; }
}  // namespace fc
