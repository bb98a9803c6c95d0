// fp32 K/V instantiations of the attend kernel.
#include "mac_attend.cuh"

namespace mac {
cudaError_t launch_attend_f32(const AttendParams &p, int G, int grid, cudaStream_t s) {
  return launch_attend_t<float>(p, G, grid, s);
}
int attend_occupancy_f32(int G, bool paged, int n_units) {
  return occupancy_t<float>(G, paged, n_units);
}
}  // namespace mac
