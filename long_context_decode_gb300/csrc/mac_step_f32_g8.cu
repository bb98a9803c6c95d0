// Step-kernel instantiations: f32 K/V and queries, 8 query head(s) per KV head.
#include "mac_step_launch.cuh"

MAC_STEP_UNIT(float, f32, 8)
