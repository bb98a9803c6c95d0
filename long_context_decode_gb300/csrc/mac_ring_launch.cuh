// Launch helpers of the ring kernel, instantiated per element type in
// mac_ring_{bf16,f32}_g8.cu (one translation unit each, so the builds run
// in parallel).
#pragma once

#include "mac_ring.cuh"

namespace mac {
namespace ring {

// per device: the dynamic shared memory limit set on the kernel (0: not yet)
template <typename T, int G, bool PAGED>
static size_t &step_smem_limit(int dev) {
  static size_t limit[64] = {0};
  return limit[dev];
}

template <typename T, int G, bool PAGED>
static cudaError_t prepare_step(int U, int B, size_t *smem) {
  using S = Step<T, G, PAGED>;
  *smem = S::smem_bytes(U, B);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && step_smem_limit<T, G, PAGED>(dev) == 0) {
    // the opt-in maximum per block, less the kernel's static shared memory
    int optin = 0;
    cudaFuncAttributes fa;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess ||
        (e = cudaFuncGetAttributes(&fa, step_kernel<T, G, PAGED>)) != cudaSuccess)
      return e;
    size_t dyn = (size_t)optin - fa.sharedSizeBytes;
    if (dyn > kMaxSmem) dyn = kMaxSmem;
    e = cudaFuncSetAttribute(step_kernel<T, G, PAGED>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
    if (e != cudaSuccess) return e;
    step_smem_limit<T, G, PAGED>(dev) = dyn;
  }
  if (dev < 64 && *smem > step_smem_limit<T, G, PAGED>(dev)) return cudaErrorInvalidValue;
  return cudaSuccess;
}

// Cooperative launch: the grid (one CTA per SM) is guaranteed co-resident,
// which the grid barrier and the long-band counts of the step rely on.
template <typename T, int G, bool PAGED>
static cudaError_t launch_step_g(const StepParams &p_in, int grid, cudaStream_t s) {
  using S = Step<T, G, PAGED>;
  size_t smem = 0;
  cudaError_t e = prepare_step<T, G, PAGED>(p_in.B * p_in.Hkv, p_in.B, &smem);
  if (e != cudaSuccess) return e;
  // the warps' query entries, where shared memory allows them
  StepParams p = p_in;
  int dev = 0;
  cudaGetDevice(&dev);
  const size_t with_q = smem + (size_t)S::kQBuf;
  p.qslot = dev < 64 && with_q <= step_smem_limit<T, G, PAGED>(dev) ? 1 : 0;
  if (p.qslot) smem = with_q;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, step_kernel<T, G, PAGED>, p);
}

template <typename T, int G, bool PAGED>
static int occupancy_g(int U, int B) {
  size_t smem = 0;
  if (prepare_step<T, G, PAGED>(U, B, &smem) != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, step_kernel<T, G, PAGED>, kThreads, smem) != cudaSuccess)
    return 0;
  return n;
}

}  // namespace ring
}  // namespace mac

// One translation unit: element type T (name TN) and group size G.
#define MAC_RING_UNIT(T, TN, G)                                                                         \
  namespace mac {                                                                                       \
  namespace ring {                                                                                      \
  cudaError_t launch_##TN##_g##G(const StepParams &p, int grid, cudaStream_t s) {                       \
    return p.kv.paged ? launch_step_g<T, G, true>(p, grid, s) : launch_step_g<T, G, false>(p, grid, s); \
  }                                                                                                     \
  int occupancy_##TN##_g##G(bool paged, int U, int B) {                                                 \
    return paged ? occupancy_g<T, G, true>(U, B) : occupancy_g<T, G, false>(U, B);                     \
  }                                                                                                     \
  }                                                                                                     \
  }
