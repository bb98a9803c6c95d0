// mac_append.cu -- Rectify-append ([MAC] "Paper version: K1/K2/K3", K3):
// slot pos mod K of every (request, head) ring <- (pos, q~, AS_{1:pos-r}).
// The rectified summary was accumulated by the step kernel as the cached
// part plus the fresh tokens up to m-r, so appending is a copy.  It runs on
// the caller's auxiliary stream after an event; the next step on the same
// rings waits for it.
#include "mac_common.cuh"

namespace mac {

template <typename T>
__global__ void __launch_bounds__(64) append_kernel(const __grid_constant__ AppendParams p) {
  constexpr int PER = 16 / (int)sizeof(T);
  const int bh = blockIdx.x, b = bh / p.Hq, h = bh % p.Hq;
  const int64_t pos = (int64_t)p.pos_base[b] + p.pos_add;
  if (pos < 1 || pos > p.capacity) return;
  const int64_t slot = (int64_t)bh * p.K + pos % p.K;
  const uint4 *qs = reinterpret_cast<const uint4 *>(p.q_src) + ((int64_t)bh * p.q_stride + p.q_offset) / PER;
  uint4 *qd = reinterpret_cast<uint4 *>(p.ring_q) + slot * (kHeadDim / PER);
  for (int i = threadIdx.x; i < kHeadDim / PER; i += blockDim.x) qd[i] = qs[i];
  const float4 *os = reinterpret_cast<const float4 *>(p.src_o + (int64_t)bh * kHeadDim);
  float4 *od = reinterpret_cast<float4 *>(p.ring_o + slot * kHeadDim);
  for (int i = threadIdx.x; i < kHeadDim / 4; i += blockDim.x) od[i] = os[i];
  if (threadIdx.x == 0) {
    p.ring_lse[slot] = p.src_lse[bh];
    if (h == 0) p.ring_pos[(int64_t)b * p.K + pos % p.K] = (int32_t)pos;
  }
}

// The ready gate: a request whose flag is set starts over with an empty
// ring (no slot holds a position, so its next step has no candidate, misses
// on every head and attends [1, m] exactly; the appends then refill the
// ring).  The flag is consumed.  One CTA per request.
__global__ void __launch_bounds__(256) reset_kernel(int32_t *ring_pos, int32_t *flags, int K) {
  const int b = blockIdx.x;
  if (flags[b] == 0) return;  // the same value in every thread of the CTA
  for (int s = threadIdx.x; s < K; s += blockDim.x) ring_pos[(int64_t)b * K + s] = 0;
  __syncthreads();  // every thread has read the flag
  if (threadIdx.x == 0) flags[b] = 0;
}

cudaError_t launch_reset(int32_t *ring_pos, int32_t *flags, int B, int K, cudaStream_t s) {
  reset_kernel<<<B, 256, 0, s>>>(ring_pos, flags, K);
  return cudaGetLastError();
}

cudaError_t launch_append(const AppendParams &p, int dtype, cudaStream_t s) {
  if (dtype == MAC_BF16)
    append_kernel<uint16_t><<<p.B * p.Hq, 64, 0, s>>>(p);
  else
    append_kernel<float><<<p.B * p.Hq, 64, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace mac
