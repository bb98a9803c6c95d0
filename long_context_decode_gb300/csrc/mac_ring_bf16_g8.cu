// Ring-kernel instantiations: bf16 K/V and queries, 8 query heads per KV head.
#include "mac_ring_launch.cuh"

MAC_RING_UNIT(uint16_t, bf16, 8)
