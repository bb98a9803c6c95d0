// bf16 instantiations of the step kernel with the phase trace compiled in
// (mac_set_trace), without front-sink pieces.
#include "mac_step_launch.cuh"

namespace mac {
cudaError_t launch_step_bf16_trace(const StepParams &p, int grid, cudaStream_t s) {
  return launch_step_t<uint16_t, false, true>(p, grid, s);
}
}  // namespace mac
