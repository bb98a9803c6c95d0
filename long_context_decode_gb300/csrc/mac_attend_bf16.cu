// bf16 K/V instantiations of the attend kernel.
#include "mac_attend.cuh"

namespace mac {
cudaError_t launch_attend_bf16(const AttendParams &p, int G, int grid, cudaStream_t s) {
  return launch_attend_t<uint16_t>(p, G, grid, s);
}
int attend_occupancy_bf16(int G, bool paged, int n_units) {
  return occupancy_t<uint16_t>(G, paged, n_units);
}
}  // namespace mac
