// Step-kernel instantiations: bf16 K/V and queries, 8 query head(s) per KV head.
#include "mac_step_launch.cuh"

MAC_STEP_UNIT(uint16_t, bf16, 8)
