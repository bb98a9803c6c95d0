// mac_match.cu -- Match step, plus the small RoPE and rectify-append kernels.
//
// Match ([MAC] "Match (2)", "Match (3)", K1 of "Paper version: K1/K2/K3"):
// for every (request, query head) a streaming squared-L2 nearest-neighbour
// scan of the pre-RoPE query against the ring entries whose position lies in
// [m-K, m-1].  The pages expand d2 = |a|^2 + |b|^2 - 2 a.b; that form cancels
// badly for close pairs, so each lane instead sums (a-b)^2 of its elements
// (a-b of two bf16 values is exact in fp32) in a pairwise tree and the lanes
// of a slot finish the tree with shuffles: the sum carries at most ~8 roundings
// (relative error <= 8 * 2^-24), which keeps the accept/argmin decisions equal
// to the exact ones outside a 1e-6 relative band.  A tile of slots is scanned
// per CTA; within a warp the argmin is a shuffle reduction (no barrier), then
// the warps of a head and the CTAs of a (request, kv-head) unit are combined
// under one total order (smaller distance, then more recent position), so the
// result does not depend on scheduling.  The last CTA of a unit (counted with
// an atomic) turns the minima into decisions and the unit's fresh-range start.
#include "mac_common.cuh"

namespace mac {

// 16 bytes of elements -> floats (8 bf16 or 4 fp32).
template <typename T>
__device__ __forceinline__ void unpack16(const uint4 &u, float *f);
template <>
__device__ __forceinline__ void unpack16<uint16_t>(const uint4 &u, float *f) {
  f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x); f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
  f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z); f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
}
template <>
__device__ __forceinline__ void unpack16<float>(const uint4 &u, float *f) {
  f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
}

template <typename T>
__global__ void __launch_bounds__(kThreads) match_kernel(const __grid_constant__ MatchParams p) {
  constexpr int PER = 16 / (int)sizeof(T);   // elements per lane per slot (one 16-byte load)
  constexpr int LPS = kHeadDim / PER;        // lanes per slot: 16 (bf16) or 32 (fp32)
  constexpr int SPW = 32 / LPS;              // slots per warp per step
  constexpr int U = 4;                       // independent slot loads in flight per lane

  __shared__ float s_bd[kWarps];
  __shared__ int s_bp[kWarps];
  __shared__ int s_lo[kWarps];
  __shared__ int s_last;

  const int split = blockIdx.x, unit = blockIdx.y;
  const int b = unit / p.Hkv, g = unit % p.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wph = kWarps / p.G;  // warps per head
  const int hl = warp / wph, wi = warp % wph;
  const int h = g * p.G + hl;
  const int64_t bh = (int64_t)b * p.Hq + h;
  const int64_t m = p.seq_len[b];
  const bool m_ok = m >= 1 && m <= p.capacity;

  if (split == 0) {
    // stage the pre-RoPE queries of the unit for the append, and rotate them
    // into q_rot for the attention (R(m) q~ * log2(e)/sqrt(d))
    if (tid == 0 && !m_ok) set_status(p.ctl, MAC_DEV_BAD_SEQ_LEN);
    const int n16 = p.G * kHeadDim / PER;
    const uint4 *src = reinterpret_cast<const uint4 *>(p.q_pre) + (int64_t)b * p.Hq * kHeadDim / PER +
                       (int64_t)g * p.G * kHeadDim / PER;
    uint4 *dst = reinterpret_cast<uint4 *>(p.stage_q) + (int64_t)b * p.Hq * kHeadDim / PER +
                 (int64_t)g * p.G * kHeadDim / PER;
    for (int i = tid; i < n16; i += kThreads) dst[i] = src[i];
    for (int idx = tid; idx < p.G * (kHeadDim / 2); idx += kThreads) {
      const int hh = idx / (kHeadDim / 2), j = idx % (kHeadDim / 2);
      const int64_t bhh = (int64_t)b * p.Hq + g * p.G + hh;
      if (!rope_rotate_pair<T>(p.q_pre, bhh * kHeadDim, p.q_rot + bhh * kHeadDim, j, m, p.rope_mode,
                               p.rope_w[j], p.q_scale))
        set_status(p.ctl, MAC_DEV_NONFINITE_Q);
    }
  }

  // this lane's piece of the current query
  const int sub = lane % LPS, sg = lane / LPS;
  float qv[PER];
  unpack16<T>(reinterpret_cast<const uint4 *>(p.q_pre)[bh * (kHeadDim / PER) + sub], qv);

  const int s0 = (int)((int64_t)p.K * split / p.n_splits);
  const int s1 = (int)((int64_t)p.K * (split + 1) / p.n_splits);
  const int64_t pos_lo = (m - p.K) > 1 ? (m - p.K) : 1;
  const int64_t pos_hi = m - 1;
  const int stride = wph * SPW;
  const uint4 *ring = reinterpret_cast<const uint4 *>(p.ring_q) + bh * (int64_t)p.K * (kHeadDim / PER);
  const int32_t *rpos = p.ring_pos + (int64_t)b * p.K;

  float bd = INFINITY;
  int bp = -1;
  // `base` is warp-uniform, so every lane runs the same iterations (the
  // shuffles below need the whole warp); slots past s1 load nothing.
  for (int base = s0 + wi * SPW; base < s1; base += stride * U) {
    uint4 u[U];
    int pos[U];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int ss = base + sg + j * stride;
      if (ss < s1) {
        u[j] = __ldcs(ring + (int64_t)ss * (kHeadDim / PER) + sub);
        pos[j] = rpos[ss];
      } else {
        u[j] = make_uint4(0, 0, 0, 0);
        pos[j] = 0;
      }
    }
#pragma unroll
    for (int j = 0; j < U; ++j) {
      float e[PER];
      unpack16<T>(u[j], e);
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const float df = __fsub_rn(qv[i], e[i]);  // exact for two bf16 values
        e[i] = __fmul_rn(df, df);
      }
      // pairwise tree inside the lane
#pragma unroll
      for (int w2 = PER / 2; w2 >= 1; w2 >>= 1)
#pragma unroll
        for (int i = 0; i < w2; ++i) e[i] = __fadd_rn(e[i], e[i + w2]);
      float D = e[0];
      // ... finished across the lanes of the slot
#pragma unroll
      for (int off = LPS / 2; off >= 1; off >>= 1) D = __fadd_rn(D, __shfl_xor_sync(0xffffffffu, D, off));
      const int ps = pos[j];
      const bool valid = m_ok && ps >= pos_lo && ps <= pos_hi;
      if (valid && better(D, ps, bd, bp)) {
        bd = D;
        bp = ps;
      }
    }
  }
  // combine the slot groups of the warp, then the warps of the head
#pragma unroll
  for (int off = 16; off >= LPS; off >>= 1) {
    const float d2 = __shfl_xor_sync(0xffffffffu, bd, off);
    const int p2 = __shfl_xor_sync(0xffffffffu, bp, off);
    if (better(d2, p2, bd, bp)) {
      bd = d2;
      bp = p2;
    }
  }
  if (lane == 0) {
    s_bd[warp] = bd;
    s_bp[warp] = bp;
  }
  __syncthreads();
  if (wi == 0 && lane == 0) {
    for (int w = warp + 1; w < warp + wph; ++w)
      if (better(s_bd[w], s_bp[w], bd, bp)) {
        bd = s_bd[w];
        bp = s_bp[w];
      }
    p.match_part[bh * kMaxSplits + split] = make_int2(__float_as_int(bd), bp);
  }

  // the last CTA of the unit turns the per-split minima into decisions
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(&p.match_cnt[unit], 1) == p.n_splits - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (wi == 0) {
    float d = INFINITY;
    int pp = -1;
    for (int i = lane; i < p.n_splits; i += 32) {
      const int2 e = __ldcg(&p.match_part[bh * kMaxSplits + i]);
      const float de = __int_as_float(e.x);
      if (better(de, e.y, d, pp)) {
        d = de;
        pp = e.y;
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const float d2 = __shfl_xor_sync(0xffffffffu, d, off);
      const int p2 = __shfl_xor_sync(0xffffffffu, pp, off);
      if (better(d2, p2, d, pp)) {
        d = d2;
        pp = p2;
      }
    }
    if (lane == 0) {
      // strict acceptance below the squared threshold ([MAC] K1: miss if d2 >= thr^2)
      const bool hit = m_ok && pp >= 1 && d < p.thr2 && m >= p.min_context;
      const int lo = hit ? (pp - p.r + 1 > 1 ? pp - p.r + 1 : 1) : 1;
      p.head_info[bh] = make_int2(hit ? pp : -1, lo);
      if (p.match_pos_out) p.match_pos_out[bh] = hit ? pp : -1;
      s_lo[hl] = lo;
    }
  }
  __syncthreads();
  if (tid == 0) {
    int s = 0x7fffffff;
    for (int i = 0; i < p.G; ++i) s = s_lo[i] < s ? s_lo[i] : s;
    p.unit_s[unit] = s;
    p.match_cnt[unit] = 0;
  }
}

// R(pos) q~ for full attention (pos = m) and for seeding (pos = the seeded
// position, summary length pos - r).
template <typename T>
__global__ void __launch_bounds__(64) rope_kernel(const __grid_constant__ RopeParams p) {
  const int bh = blockIdx.x, b = bh / p.Hq, h = bh % p.Hq;
  const int64_t pos = (int64_t)p.pos_base[b] + p.pos_add;
  const int64_t src = p.n_seed > 0 ? ((int64_t)bh * p.n_seed + p.seed_index) * kHeadDim
                                   : (int64_t)bh * kHeadDim;
  for (int j = threadIdx.x; j < kHeadDim / 2; j += blockDim.x) {
    if (!rope_rotate_pair<T>(p.q, src, p.q_rot + (int64_t)bh * kHeadDim, j, pos, p.rope_mode,
                             p.rope_w[j], p.q_scale))
      set_status(p.ctl, MAC_DEV_NONFINITE_Q);
  }
  if (p.seed_pos && h == 0 && threadIdx.x == 0) {
    p.seed_pos[b] = pos >= 1 ? (int32_t)pos : 0;
    p.seed_len[b] = pos >= 1 ? (int32_t)(pos - p.r) : 0;
  }
}

// Rectify-append ([MAC] K3): slot pos mod K <- (pos, q~, AS_{1:pos-r}).
template <typename T>
__global__ void __launch_bounds__(64) append_kernel(const __grid_constant__ AppendParams p) {
  const int bh = blockIdx.x, b = bh / p.Hq, h = bh % p.Hq;
  const int64_t pos = p.pos[b];
  if (pos < 1 || pos > p.capacity) return;
  const int64_t slot = (int64_t)bh * p.K + pos % p.K;
  constexpr int PER = 16 / (int)sizeof(T);
  const int64_t src = p.n_seed > 0 ? ((int64_t)bh * p.n_seed + p.seed_index) * kHeadDim
                                   : (int64_t)bh * kHeadDim;
  const uint4 *qs = reinterpret_cast<const uint4 *>(p.q_src) + src / PER;
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

cudaError_t launch_match(const MatchParams &p, int dtype, cudaStream_t s) {
  dim3 grid(p.n_splits, p.B * p.Hkv);
  if (dtype == MAC_BF16)
    match_kernel<uint16_t><<<grid, kThreads, 0, s>>>(p);
  else
    match_kernel<float><<<grid, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_rope(const RopeParams &p, int dtype, cudaStream_t s) {
  if (dtype == MAC_BF16)
    rope_kernel<uint16_t><<<p.B * p.Hq, 64, 0, s>>>(p);
  else
    rope_kernel<float><<<p.B * p.Hq, 64, 0, s>>>(p);
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
