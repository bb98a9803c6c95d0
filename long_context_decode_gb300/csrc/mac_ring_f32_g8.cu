// Ring-kernel instantiations: f32 K/V and queries, 8 query heads per KV head.
#include "mac_ring_launch.cuh"

MAC_RING_UNIT(float, f32, 8)
