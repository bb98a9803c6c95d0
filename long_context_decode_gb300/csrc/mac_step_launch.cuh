// Launch helpers of the step kernel, instantiated once per element type and
// front-sink variant in mac_step_{bf16,f32}{,_sink}.cu, and once with the
// phase trace in mac_step_bf16_trace.cu (one translation unit each, so the
// builds run in parallel).
#pragma once

#include "mac_step.cuh"

namespace mac {

template <typename T, int G, bool PAGED, bool SINK, bool TRACE>
static cudaError_t prepare_step(int B, int Hq, int Hkv, int K, size_t *smem) {
  using S = Step<T, G, PAGED, SINK, TRACE>;
  *smem = S::smem_bytes(B, Hq, Hkv, K);
  static size_t limit[64] = {0};  // per device: dynamic shared memory limit set on the kernel
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && limit[dev] == 0) {
    // the opt-in maximum per block, less the kernel's static shared memory
    int optin = 0;
    cudaFuncAttributes fa;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess ||
        (e = cudaFuncGetAttributes(&fa, step_kernel<T, G, PAGED, SINK, TRACE>)) != cudaSuccess)
      return e;
    size_t dyn = (size_t)optin - fa.sharedSizeBytes;
    if (dyn > kMaxSmem) dyn = kMaxSmem;
    e = cudaFuncSetAttribute(step_kernel<T, G, PAGED, SINK, TRACE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn);
    if (e != cudaSuccess) return e;
    limit[dev] = dyn;
  }
  if (dev < 64 && *smem > limit[dev]) return cudaErrorInvalidValue;
  return cudaSuccess;
}

// Cooperative launch: the grid (one CTA per SM) is guaranteed co-resident,
// which the grid barriers of the step rely on.
template <typename T, int G, bool PAGED, bool SINK, bool TRACE>
static cudaError_t launch_step_g(const StepParams &p, int grid, cudaStream_t s) {
  size_t smem = 0;
  cudaError_t e = prepare_step<T, G, PAGED, SINK, TRACE>(p.B, p.Hq, p.Hkv, p.K, &smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (p.early_start) {
    // An early start: the CTAs may begin on the SMs the previous step kernel
    // frees (griddep_wait in the kernel orders everything that depends on
    // it).  A cooperative launch would place no CTA before the whole grid
    // fits, so this one is plain: the grid (one CTA per SM, which its shared
    // memory enforces) is resident once the previous kernel has finished,
    // and the grid barrier's wait is bounded should another stream hold SMs.
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
  } else {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, step_kernel<T, G, PAGED, SINK, TRACE>, p);
}

template <typename T, int G, bool PAGED, bool SINK, bool TRACE>
static int occupancy_g(int B, int Hq, int Hkv, int K) {
  size_t smem = 0;
  if (prepare_step<T, G, PAGED, SINK, TRACE>(B, Hq, Hkv, K, &smem) != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, step_kernel<T, G, PAGED, SINK, TRACE>, kThreads, smem) !=
      cudaSuccess)
    return 0;
  return n;
}

template <typename T, bool SINK, bool TRACE>
static cudaError_t launch_step_t(const StepParams &p, int grid, cudaStream_t s) {
  const bool paged = p.kv.paged != 0;
  switch (p.G) {
    case 1: return paged ? launch_step_g<T, 1, true, SINK, TRACE>(p, grid, s) : launch_step_g<T, 1, false, SINK, TRACE>(p, grid, s);
    case 2: return paged ? launch_step_g<T, 2, true, SINK, TRACE>(p, grid, s) : launch_step_g<T, 2, false, SINK, TRACE>(p, grid, s);
    case 4: return paged ? launch_step_g<T, 4, true, SINK, TRACE>(p, grid, s) : launch_step_g<T, 4, false, SINK, TRACE>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T, bool SINK, bool TRACE>
static int occupancy_t(int G, bool paged, int B, int Hq, int Hkv, int K) {
  switch (G) {
    case 1: return paged ? occupancy_g<T, 1, true, SINK, TRACE>(B, Hq, Hkv, K) : occupancy_g<T, 1, false, SINK, TRACE>(B, Hq, Hkv, K);
    case 2: return paged ? occupancy_g<T, 2, true, SINK, TRACE>(B, Hq, Hkv, K) : occupancy_g<T, 2, false, SINK, TRACE>(B, Hq, Hkv, K);
    case 4: return paged ? occupancy_g<T, 4, true, SINK, TRACE>(B, Hq, Hkv, K) : occupancy_g<T, 4, false, SINK, TRACE>(B, Hq, Hkv, K);
    default: return 0;
  }
}

}  // namespace mac
