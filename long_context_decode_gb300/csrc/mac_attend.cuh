// mac_attend.cuh -- Complete step: span-balanced split-K decode attention of
// the post-RoPE query over each (request, kv-head) unit's fresh range, with
// the fixed-order log-domain merge of the chunk partials and the cached
// rectified summary done by the last CTA that finishes an item of the unit.
//
// [MAC] "Paper version: K1/K2/K3": K2 flattens the (request, head) axis and
// gives work in proportion to each head's band+tail span; here the span of a
// GQA group is cut into chunks (see plan_unit) and a persistent grid pulls
// chunks from one list, so long spans (misses) get many CTAs and short ones
// (hits) few.  A group loads each K/V tile once for all its query heads
// ([MAC] "GQA intra-group skew"); heads that reuse from a later position mask
// the tokens before their own band start.  [MAC] "Complete": summaries keep a
// running max and merge in log domain (base-2 here: logits are pre-scaled by
// log2 e).  K/V tiles move global -> shared with 1-D TMA bulk copies into a
// kStages-deep ring of buffers completed on mbarriers.
#pragma once

#include "mac_common.cuh"

namespace mac {

template <typename T>
struct Pieces;
template <>
struct Pieces<uint16_t> {  // bf16: 8 elements per 16-byte piece, 2 pieces per lane
  static constexpr int kPer = 8, kN = 2;
  __device__ static void unpack(const uint4 &u, float *f) {
    f[0] = bf16_lo(u.x); f[1] = bf16_hi(u.x); f[2] = bf16_lo(u.y); f[3] = bf16_hi(u.y);
    f[4] = bf16_lo(u.z); f[5] = bf16_hi(u.z); f[6] = bf16_lo(u.w); f[7] = bf16_hi(u.w);
  }
};
template <>
struct Pieces<float> {  // fp32: 4 elements per piece, 4 pieces per lane
  static constexpr int kPer = 4, kN = 4;
  __device__ static void unpack(const uint4 &u, float *f) {
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
  }
};

// Lane `sub` (0..7) of a token's 8-lane group owns 16 dimensions: piece c
// covers dims [c*8*kPer + sub*kPer, +kPer).  Each 8-lane group thus reads 128
// contiguous bytes of a row per piece (no shared-memory bank conflicts).
template <typename T>
__device__ __forceinline__ int piece_dim(int c, int sub) {
  return c * 8 * Pieces<T>::kPer + sub * Pieces<T>::kPer;
}

// (M, L, O) <- (M, L, O) (+) (m2, l2, o2) in base-2 log domain; an empty
// operand (L == 0) is the identity.
__device__ __forceinline__ void merge_scalar(float &M, float &L, float &O, float m2, float l2,
                                             float o2) {
  if (l2 == 0.f) return;
  if (L == 0.f) {
    M = m2;
    L = l2;
    O = o2;
    return;
  }
  float mn = fmaxf(M, m2);
  float a = ex2(M - mn), c = ex2(m2 - mn);
  L = L * a + l2 * c;
  O = O * a + o2 * c;
  M = mn;
}

template <typename T, int G, bool PAGED>
struct Attend {
  static constexpr int kRowBytes = kHeadDim * (int)sizeof(T);
  static constexpr int kTileBytes = kTile * kRowBytes;
  static constexpr int kPer = Pieces<T>::kPer;
  static constexpr int kNP = Pieces<T>::kN;

  static constexpr size_t kKvBytes = (size_t)kStages * 2 * kTileBytes;
  static constexpr size_t kRedBytes = (size_t)kWarps * G * kPartStride * sizeof(float);
  static size_t smem_bytes(int n_units) {
    return kKvBytes + 64 + kRedBytes + sizeof(int32_t) * (size_t)(n_units + 1);
  }

  // Issue the TMA copies of the rows of tile `tile` (tokens [tile*kTile+1,
  // tile*kTile+kTile]) that fall in [lo, hi], each to its fixed row of the
  // stage buffers, so no byte outside the chunk is read.  *mask records which
  // 16-token halves hold valid data.  Called by one thread.
  __device__ static void issue_tile(const AttendParams &p, int b, int g, int64_t lo, int64_t hi,
                                    int64_t tile, uint8_t *kbuf, uint8_t *vbuf, uint32_t bar,
                                    int *mask) {
    const int64_t t0 = tile * kTile;  // tokens t0+1 .. t0+kTile
    if (!PAGED) {
      int64_t a = t0 + 1 > lo ? t0 + 1 : lo;
      int64_t z = t0 + kTile < hi ? t0 + kTile : hi;
      size_t off = (((size_t)b * p.Hkv + g) * (size_t)p.kv.capacity + (size_t)(a - 1)) * kRowBytes;
      uint32_t bytes = (uint32_t)(z - a + 1) * kRowBytes;
      uint32_t dst = (uint32_t)(a - t0 - 1) * kRowBytes;
      *mask = 3;
      mbar_expect_tx(bar, 2 * bytes);
      bulk_g2s(smem_addr(kbuf + dst), (const uint8_t *)p.kv.k + off, bytes, bar);
      bulk_g2s(smem_addr(vbuf + dst), (const uint8_t *)p.kv.v + off, bytes, bar);
    } else {
      int32_t pid[2];
      int64_t ra[2], rz[2];
      int msk = 0;
      uint32_t bytes = 0;
      for (int pg = 0; pg < 2; ++pg) {
        const int64_t slot = tile * 2 + pg;
        const int64_t pa = t0 + pg * 16 + 1, pz = pa + 15;
        ra[pg] = pa > lo ? pa : lo;
        rz[pg] = pz < hi ? pz : hi;
        pid[pg] = -1;
        if (ra[pg] > rz[pg] || slot >= p.kv.max_pages) continue;
        const int32_t id = p.kv.page_table[(int64_t)b * p.kv.max_pages + slot];
        if (id < 0 || id >= p.kv.n_pages) {
          set_status(p.ctl, MAC_DEV_BAD_PAGE);
          continue;
        }
        pid[pg] = id;
        msk |= 1 << pg;
        bytes += (uint32_t)(rz[pg] - ra[pg] + 1) * kRowBytes;
      }
      *mask = msk;
      if (bytes == 0) {
        mbar_arrive(bar);
        return;
      }
      mbar_expect_tx(bar, 2 * bytes);
      for (int pg = 0; pg < 2; ++pg) {
        if (pid[pg] < 0) continue;
        const int64_t in_page = (ra[pg] - 1) % 16;
        const size_t off = (((size_t)pid[pg] * p.Hkv + g) * 16 + (size_t)in_page) * kRowBytes;
        const uint32_t nbytes = (uint32_t)(rz[pg] - ra[pg] + 1) * kRowBytes;
        const uint32_t dst = (uint32_t)(ra[pg] - t0 - 1) * kRowBytes;
        bulk_g2s(smem_addr(kbuf + dst), (const uint8_t *)p.kv.k + off, nbytes, bar);
        bulk_g2s(smem_addr(vbuf + dst), (const uint8_t *)p.kv.v + off, nbytes, bar);
      }
    }
  }

  __device__ static int64_t unit_start(const AttendParams &p, int u) {
    return p.mode == MODE_DECODE ? (int64_t)p.unit_s[u] : 1;
  }

  // The scratch holds the chunk partials of lengths up to max_len only.
  __device__ static bool len_ok(const AttendParams &p, int64_t m) {
    return m >= 1 && m <= p.max_len;
  }

  __device__ static UnitPlan plan(const AttendParams &p, int u) {
    int b = u / p.Hkv;
    int64_t m = p.len[b];
    if (!len_ok(p, m)) return plan_unit(0, 1, p.r);
    return plan_unit(m, unit_start(p, u), p.r);
  }

  // prefix[u] = first item of unit u; prefix[n_units] = total items.
  __device__ static void build_prefix(const AttendParams &p, int32_t *prefix, int n_units) {
    __shared__ int wsum[kWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int seg = (n_units + kThreads - 1) / kThreads;
    const int beg = tid * seg;
    const int end = min(beg + seg, n_units);
    int run = 0;
    for (int u = beg; u < end; ++u) {
      run += plan(p, u).n_items;
      prefix[u + 1] = run;
    }
    int x = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = lane < kWarps ? wsum[lane] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, w, off);
        if (lane >= off) w += y;
      }
      if (lane < kWarps) wsum[lane] = w;
    }
    __syncthreads();
    int excl = x - run + (warp > 0 ? wsum[warp - 1] : 0);
    for (int u = beg; u < end; ++u) prefix[u + 1] += excl;
    if (tid == 0) prefix[0] = 0;
    __syncthreads();
  }

  // Merge the unit's chunk partials (and, when decoding, the cached summary)
  // in item order; write AS_{1:m-r} after the band items and the output.
  __device__ static void merge_unit(const AttendParams &p, int u, int first_item,
                                    const UnitPlan &up) {
    const int b = u / p.Hkv, g = u % p.Hkv;
    const int n = up.n_items;
    const int nb = (up.nb + up.nt == 0) ? n : up.nb;
    for (int idx = threadIdx.x; idx < G * kHeadDim; idx += kThreads) {
      const int hh = idx / kHeadDim, dim = idx % kHeadDim;
      const int64_t bh = (int64_t)b * p.Hq + g * G + hh;
      float M = -INFINITY, L = 0.f, O = 0.f;
      if (p.mode == MODE_DECODE) {
        int2 hi = p.head_info[bh];
        if (hi.x >= 1) {
          int64_t slot = bh * p.K + hi.x % p.K;
          float lse = p.ring_lse[slot];
          if (lse > -INFINITY) {
            M = lse * kLog2e;
            L = 1.f;
            O = p.ring_o[slot * kHeadDim + dim];
          }
        }
      }
      const float *part = p.partials + ((int64_t)first_item * G + hh) * kPartStride;
      for (int i0 = 0; i0 < n; i0 += 4) {
        float pm[4], pl[4], po[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (i0 + j < n) {
            const float *pp = part + (int64_t)(i0 + j) * G * kPartStride;
            pm[j] = __ldcg(pp + kHeadDim);
            pl[j] = __ldcg(pp + kHeadDim + 1);
            po[j] = __ldcg(pp + dim);
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          int i = i0 + j;
          if (i >= n) break;
          if (i == nb && p.mode == MODE_DECODE && p.as_o) {
            p.as_o[bh * kHeadDim + dim] = L > 0.f ? O / L : 0.f;
            if (dim == 0) p.as_lse[bh] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
          }
          merge_scalar(M, L, O, pm[j], pl[j], po[j]);
        }
      }
      if (nb == n && p.mode == MODE_DECODE && p.as_o) {
        p.as_o[bh * kHeadDim + dim] = L > 0.f ? O / L : 0.f;
        if (dim == 0) p.as_lse[bh] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
      }
      p.out[bh * kHeadDim + dim] = L > 0.f ? O / L : 0.f;
      if (p.out_lse && dim == 0) p.out_lse[bh] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
    }
  }

  __device__ static void run(const AttendParams &p) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *kv_smem = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kKvBytes);
    float *red = reinterpret_cast<float *>(smem + kKvBytes + 64);
    int32_t *prefix = reinterpret_cast<int32_t *>(smem + kKvBytes + 64 + kRedBytes);
    __shared__ int s_item, s_last;
    __shared__ int s_mask[kStages];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int lg = lane >> 3, sub = lane & 7;
    const int row = warp * 4 + lg;  // token row of this lane group inside a tile
    const int n_units = p.B * p.Hkv;

    if (tid == 0) {
      for (int i = 0; i < kStages; ++i) mbar_init(smem_addr(&bars[i]), 1);
      mbar_fence_init();
    }
    build_prefix(p, prefix, n_units);  // ends with __syncthreads
    const int total = prefix[n_units];
    uint32_t parity = 0;
    bool aborted = false;  // a bounded wait gave up: stop touching the stage buffers

    for (;;) {
      if (tid == 0) s_item = atomicAdd(&p.ctl[1], 1);
      __syncthreads();
      const int item = s_item;
      if (item >= total) break;

      int lo_u = 0, hi_u = n_units - 1;
      while (lo_u < hi_u) {
        int mid = (lo_u + hi_u + 1) >> 1;
        if (prefix[mid] <= item) lo_u = mid; else hi_u = mid - 1;
      }
      const int u = lo_u;
      const int first = prefix[u];
      const int b = u / p.Hkv, g = u % p.Hkv;
      const UnitPlan up = plan(p, u);
      int64_t lo_c, hi_c;
      bool band;
      item_range(up, p.r, item - first, &lo_c, &hi_c, &band);
      if (p.check_len && tid == 0 && item == first && !len_ok(p, p.len[b]))
        set_status(p.ctl, MAC_DEV_BAD_SEQ_LEN);

      int64_t lo_h[G];
      float q[G][16], o[G][16], mrun[G], lrun[G];
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        const int64_t bh = (int64_t)b * p.Hq + g * G + hh;
        lo_h[hh] = p.mode == MODE_DECODE ? (int64_t)p.head_info[bh].y : 1;
        const float *qr = p.q_rot + bh * kHeadDim;
#pragma unroll
        for (int c = 0; c < kNP; ++c) {
#pragma unroll
          for (int e4 = 0; e4 < kPer; e4 += 4) {
            float4 v = *reinterpret_cast<const float4 *>(qr + piece_dim<T>(c, sub) + e4);
            q[hh][c * kPer + e4 + 0] = v.x;
            q[hh][c * kPer + e4 + 1] = v.y;
            q[hh][c * kPer + e4 + 2] = v.z;
            q[hh][c * kPer + e4 + 3] = v.w;
          }
        }
        mrun[hh] = -INFINITY;
        lrun[hh] = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) o[hh][i] = 0.f;
      }

      if (lo_c <= hi_c && !aborted) {
        const int64_t tile_first = (lo_c - 1) / kTile;
        const int ntiles = (int)((hi_c - 1) / kTile - tile_first + 1);
        if (tid == 0) {
          for (int k = 0; k < kStages && k < ntiles; ++k) {
            uint8_t *kb = kv_smem + (size_t)k * 2 * kTileBytes;
            fence_proxy_async();
            issue_tile(p, b, g, lo_c, hi_c, tile_first + k, kb, kb + kTileBytes,
                       smem_addr(&bars[k]), &s_mask[k]);
          }
        }
        for (int k = 0; k < ntiles; ++k) {
          const int st = k % kStages;
          const bool timed_out = !mbar_wait_bounded(smem_addr(&bars[st]), (parity >> st) & 1u);
          parity ^= 1u << st;
          const uint8_t *kb = kv_smem + (size_t)st * 2 * kTileBytes;
          const uint8_t *vb = kb + kTileBytes;
          const int64_t t = (tile_first + k) * kTile + row + 1;
          const bool tok = t >= lo_c && t <= hi_c && ((s_mask[st] >> (row >> 4)) & 1);

          float kf[16], vf[16];
#pragma unroll
          for (int c = 0; c < kNP; ++c) {
            uint4 uk = *reinterpret_cast<const uint4 *>(kb + row * kRowBytes + c * 128 + sub * 16);
            Pieces<T>::unpack(uk, kf + c * kPer);
          }
          float sc[G];
#pragma unroll
          for (int hh = 0; hh < G; ++hh) {
            float acc = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) acc = fmaf(q[hh][i], kf[i], acc);
            acc += __shfl_xor_sync(0xffffffffu, acc, 1);
            acc += __shfl_xor_sync(0xffffffffu, acc, 2);
            acc += __shfl_xor_sync(0xffffffffu, acc, 4);
            sc[hh] = acc;
          }
#pragma unroll
          for (int c = 0; c < kNP; ++c) {
            uint4 uv = *reinterpret_cast<const uint4 *>(vb + row * kRowBytes + c * 128 + sub * 16);
            Pieces<T>::unpack(uv, vf + c * kPer);
          }
#pragma unroll
          for (int hh = 0; hh < G; ++hh) {
            if (tok && t >= lo_h[hh]) {
              const float s = sc[hh];
              if (s > mrun[hh]) {
                const float f = ex2(mrun[hh] - s);
                lrun[hh] *= f;
#pragma unroll
                for (int i = 0; i < 16; ++i) o[hh][i] *= f;
                mrun[hh] = s;
              }
              const float w = ex2(s - mrun[hh]);
              lrun[hh] += w;
#pragma unroll
              for (int i = 0; i < 16; ++i) o[hh][i] = fmaf(w, vf[i], o[hh][i]);
            }
          }
          // stage st fully consumed; every thread learns whether any wait gave up
          if (__syncthreads_or(timed_out)) {
            if (tid == 0) set_status(p.ctl, MAC_DEV_WAIT_TIMEOUT);
            aborted = true;
            break;
          }
          if (tid == 0 && k + kStages < ntiles) {
            uint8_t *kbw = kv_smem + (size_t)st * 2 * kTileBytes;
            fence_proxy_async();
            issue_tile(p, b, g, lo_c, hi_c, tile_first + k + kStages, kbw, kbw + kTileBytes,
                       smem_addr(&bars[st]), &s_mask[st]);
          }
        }
      }

      // combine the 4 token groups of the warp (lanes differing in bits 3, 4)
#pragma unroll
      for (int off = 8; off <= 16; off <<= 1) {
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          const float m2 = __shfl_xor_sync(0xffffffffu, mrun[hh], off);
          const float l2 = __shfl_xor_sync(0xffffffffu, lrun[hh], off);
          const float mn = fmaxf(mrun[hh], m2);
          const float a = lrun[hh] > 0.f ? ex2(mrun[hh] - mn) : 0.f;
          const float c2 = l2 > 0.f ? ex2(m2 - mn) : 0.f;
          lrun[hh] = lrun[hh] * a + l2 * c2;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float o2 = __shfl_xor_sync(0xffffffffu, o[hh][i], off);
            o[hh][i] = o[hh][i] * a + o2 * c2;
          }
          mrun[hh] = (lrun[hh] > 0.f) ? mn : -INFINITY;
        }
      }
      if (lg == 0) {
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          float *rw = red + ((size_t)warp * G + hh) * kPartStride;
#pragma unroll
          for (int c = 0; c < kNP; ++c)
#pragma unroll
            for (int e = 0; e < kPer; ++e) rw[piece_dim<T>(c, sub) + e] = o[hh][c * kPer + e];
          if (sub == 0) {
            rw[kHeadDim] = mrun[hh];
            rw[kHeadDim + 1] = lrun[hh];
          }
        }
      }
      __syncthreads();
      // combine the warps in a fixed order and store the item's partial
      for (int idx = tid; idx < G * kHeadDim; idx += kThreads) {
        const int hh = idx / kHeadDim, dim = idx % kHeadDim;
        float M = -INFINITY, L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float *rw = red + ((size_t)w * G + hh) * kPartStride;
          merge_scalar(M, L, O, rw[kHeadDim], rw[kHeadDim + 1], rw[dim]);
        }
        float *dst = p.partials + ((int64_t)item * G + hh) * kPartStride;
        dst[dim] = O;
        if (dim == 0) {
          dst[kHeadDim] = M;
          dst[kHeadDim + 1] = L;
        }
      }
      __threadfence();
      __syncthreads();
      if (tid == 0) s_last = (atomicAdd(&p.unit_done[u], 1) == up.n_items - 1);
      __syncthreads();
      if (s_last) {
        __threadfence();
        merge_unit(p, u, first, up);
        __syncthreads();
        if (tid == 0) p.unit_done[u] = 0;
      }
      __syncthreads();
    }
    if (tid == 0) {
      __threadfence();
      if (atomicAdd(&p.ctl[2], 1) == (int)gridDim.x - 1) {
        p.ctl[1] = 0;
        p.ctl[2] = 0;
      }
    }
  }
};

template <typename T, int G, bool PAGED>
__global__ void __launch_bounds__(kThreads, 1) attend_kernel(const __grid_constant__ AttendParams p) {
  Attend<T, G, PAGED>::run(p);
}

}  // namespace mac

namespace mac {

// Launch / occupancy helpers, instantiated once per element type in
// mac_attend_bf16.cu and mac_attend_f32.cu (one translation unit each, so
// the builds run in parallel).
template <typename T, int G, bool PAGED>
static cudaError_t prepare_attend(int n_units, size_t *smem) {
  using A = Attend<T, G, PAGED>;
  *smem = A::smem_bytes(n_units);
  static size_t configured[64] = {0};  // per device: largest smem size already set
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && configured[dev] >= *smem) return cudaSuccess;
  e = cudaFuncSetAttribute(attend_kernel<T, G, PAGED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)A::smem_bytes(kMaxUnits));
  if (e == cudaSuccess && dev < 64) configured[dev] = A::smem_bytes(kMaxUnits);
  return e;
}

template <typename T, int G, bool PAGED>
static cudaError_t launch_attend_g(const AttendParams &p, int grid, cudaStream_t s) {
  size_t smem = 0;
  cudaError_t e = prepare_attend<T, G, PAGED>(p.B * p.Hkv, &smem);
  if (e != cudaSuccess) return e;
  attend_kernel<T, G, PAGED><<<grid, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

template <typename T, int G, bool PAGED>
static int occupancy_g(int n_units) {
  size_t smem = 0;
  if (prepare_attend<T, G, PAGED>(n_units, &smem) != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attend_kernel<T, G, PAGED>, kThreads, smem) !=
      cudaSuccess)
    return 0;
  return n;
}

template <typename T>
static cudaError_t launch_attend_t(const AttendParams &p, int G, int grid, cudaStream_t s) {
  const bool paged = p.kv.paged != 0;
  switch (G) {
    case 1: return paged ? launch_attend_g<T, 1, true>(p, grid, s) : launch_attend_g<T, 1, false>(p, grid, s);
    case 2: return paged ? launch_attend_g<T, 2, true>(p, grid, s) : launch_attend_g<T, 2, false>(p, grid, s);
    case 4: return paged ? launch_attend_g<T, 4, true>(p, grid, s) : launch_attend_g<T, 4, false>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
static int occupancy_t(int G, bool paged, int n_units) {
  switch (G) {
    case 1: return paged ? occupancy_g<T, 1, true>(n_units) : occupancy_g<T, 1, false>(n_units);
    case 2: return paged ? occupancy_g<T, 2, true>(n_units) : occupancy_g<T, 2, false>(n_units);
    case 4: return paged ? occupancy_g<T, 4, true>(n_units) : occupancy_g<T, 4, false>(n_units);
    default: return 0;
  }
}

}  // namespace mac
