// fp32 instantiations of the step kernel, with front-sink pieces.
#include "mac_step_launch.cuh"

namespace mac {
cudaError_t launch_step_f32_sink(const StepParams &p, int grid, cudaStream_t s) {
  return launch_step_t<float, true, false>(p, grid, s);
}
int step_occupancy_f32_sink(int G, bool paged, int B, int Hq, int Hkv, int K) {
  return occupancy_t<float, true, false>(G, paged, B, Hq, Hkv, K);
}
}  // namespace mac
