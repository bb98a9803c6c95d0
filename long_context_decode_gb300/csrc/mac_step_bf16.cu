// bf16 instantiations of the step kernel, without front-sink pieces.
#include "mac_step_launch.cuh"

namespace mac {
cudaError_t launch_step_bf16(const StepParams &p, int grid, cudaStream_t s) {
  return launch_step_t<uint16_t, false, false>(p, grid, s);
}
int step_occupancy_bf16(int G, bool paged, int B, int Hq, int Hkv, int K) {
  return occupancy_t<uint16_t, false, false>(G, paged, B, Hq, Hkv, K);
}
}  // namespace mac
