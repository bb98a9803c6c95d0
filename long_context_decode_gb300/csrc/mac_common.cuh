// mac_common.cuh -- internal definitions shared by the CUDA translation units
// of libmac_gb300 (never by the CPU oracle).
//
// Sources the kernels follow (section names translated):
//   [MAC]  "MAC-Attention: Match-Amend-Complete attention reuse, up to 99% fewer
//          KV reads in long-context decoding (MLSys 2026)", pinghaoyang.com.cn
//   [MACS] "MAC-Attention: A Match-Amend-Complete Scheme for Fast and Accurate
//          Attention Computation (MLSys 2026)", awesome-system-papers
//   [ACSP] "Attention Cache and Sequence Parallelism", shaojiemike.top
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "mac.h"

namespace mac {

// ---------------------------------------------------------------------------
// work decomposition constants
// ---------------------------------------------------------------------------
constexpr int kHeadDim = 128;          // supported head dimension
constexpr int kThreads = 256;          // threads per CTA (match and attend)
constexpr int kWarps = kThreads / 32;
constexpr int kTile = 32;              // tokens per K/V tile (two 16-token pages)
constexpr int kTailChunk = 128;        // tokens per tail chunk (the last r positions)
constexpr int kBandChunkMin = 128;     // band chunk size grows from here ...
constexpr int kBandChunkMax = 2048;    // ... up to here, so that a unit has at most
constexpr int kBandChunksTarget = 64;  //     kBandChunksTarget band chunks when possible
constexpr int kPartStride = kHeadDim + 4;  // floats per (item, head) partial: o[d], m, l, 0, 0
constexpr int kMaxUnits = 4096;        // B * Hkv
constexpr int kMaxSplits = 64;         // match splits per (request, kv-head) unit
constexpr int kStages = 4;             // TMA pipeline depth (tiles in flight per CTA)

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------------------
// scratch workspace (shared by the kernels of one stream)
// ---------------------------------------------------------------------------
struct ScratchLayout {
  size_t ctl;        // int32[64]: [0] status word, [1] work counter, [2] exit counter
  size_t match_part; // int2 [B][Hq][kMaxSplits]: {bits of D, position}
  size_t match_cnt;  // int32 [B*Hkv]: CTAs of the match finished per unit
  size_t head_info;  // int2 [B][Hq]: {matched position or -1, first fresh token lo}
  size_t unit_s;     // int32 [B*Hkv]: first token any head of the unit reads
  size_t q_rot;      // f32 [B][Hq][d]: R(m) q~ scaled by log2(e)/sqrt(d)
  size_t unit_done;  // int32 [B*Hkv]: items of the unit finished
  size_t seed_pos;   // int32 [B]: position being seeded
  size_t seed_len;   // int32 [B]: its summary length p - r
  size_t partials;   // f32 [max_items][G][kPartStride]
  size_t total;
  int64_t max_items;
};

// ---------------------------------------------------------------------------
// per-(request, kv-head) chunk plan
// ---------------------------------------------------------------------------
// The fresh range of a unit is [s, m] (s = first token any head of the group
// needs).  It is cut at m-r: band chunks cover [s, m-r] and end on m-r,
// tail chunks cover [m-r+1, m] in kTailChunk pieces aligned on m-r.  Every
// chunk lies wholly on one side of m-r, so per head the band chunks (plus
// the cached summary) give the rectified summary AS_{1:m-r} and the tail
// chunks complete the output ([MAC] K2/K3).  The same plan with s = 1 is the
// exact full attention, which makes a miss bitwise equal to it.
struct UnitPlan {
  int64_t m, s, t_start;
  int32_t cb, nb, j0, nt, n_items;
};

__host__ __device__ inline UnitPlan plan_unit(int64_t m, int64_t s, int r) {
  UnitPlan u;
  u.m = m;
  u.s = s;
  int64_t band_len = (m - r) - s + 1;
  u.cb = kBandChunkMin;
  if (band_len > 0) {
    while (u.cb < kBandChunkMax && (band_len + u.cb - 1) / u.cb > kBandChunksTarget) u.cb <<= 1;
    u.nb = (int32_t)((band_len + u.cb - 1) / u.cb);
  } else {
    u.nb = 0;
  }
  int64_t tail_lo = m - r + 1;
  u.t_start = s > tail_lo ? s : tail_lo;
  int32_t n_tail = (r + kTailChunk - 1) / kTailChunk;
  if (m >= 1 && u.t_start <= m && n_tail > 0) {
    u.j0 = (int32_t)((u.t_start - tail_lo) / kTailChunk);
    u.nt = n_tail - u.j0;
  } else {
    u.j0 = 0;
    u.nt = 0;
  }
  u.n_items = u.nb + u.nt > 0 ? u.nb + u.nt : 1;  // an empty unit keeps one empty item
  return u;
}

// Token range [lo, hi] of item i of the unit; band says it lies at or below m-r.
__host__ __device__ inline void item_range(const UnitPlan &u, int r, int i, int64_t *lo,
                                           int64_t *hi, bool *band) {
  if (u.nb + u.nt == 0) {
    *lo = 1;
    *hi = 0;
    *band = true;
    return;
  }
  if (i < u.nb) {
    int64_t top = (u.m - r) - (int64_t)(u.nb - 1 - i) * u.cb;
    int64_t bot = top - u.cb + 1;
    *lo = bot > u.s ? bot : u.s;
    *hi = top;
    *band = true;
  } else {
    int64_t base = u.m - r + 1 + (int64_t)(u.j0 + (i - u.nb)) * kTailChunk;
    *lo = base > u.t_start ? base : u.t_start;
    int64_t top = base + kTailChunk - 1;
    *hi = top < u.m ? top : u.m;
    *band = false;
  }
}

// Worst-case items per unit for contexts up to max_context.
__host__ inline int64_t max_items_per_unit(int64_t max_context, int r) {
  int64_t nb = kBandChunksTarget;
  int64_t by_max = (max_context + kBandChunkMax - 1) / kBandChunkMax;
  if (by_max > nb) nb = by_max;
  int64_t nt = (r + kTailChunk - 1) / kTailChunk;
  return nb + nt + 1;
}

// ---------------------------------------------------------------------------
// kernel parameter blocks
// ---------------------------------------------------------------------------
struct KvView {
  const void *k, *v;
  const int32_t *page_table;
  int64_t capacity;   // tokens per (b, g) (contiguous) or max_pages*page_size
  int32_t max_pages, n_pages, paged;
};

struct MatchParams {
  int B, Hq, Hkv, G, d, K, r, min_context, n_splits;
  float thr2;
  float q_scale;             // log2(e)/sqrt(d)
  int rope_mode;
  const void *q_pre;         // [B][Hq][d]
  const int32_t *seq_len;    // [B]
  int64_t capacity;          // max valid m: min(cache capacity, max_context)
  const int32_t *ring_pos;   // [B][K]
  const void *ring_q;        // [B][Hq][K][d]
  void *stage_q;             // [B][Hq][d]
  int32_t *ctl;
  int2 *match_part;
  int32_t *match_cnt;
  int2 *head_info;
  int32_t *unit_s;
  float *q_rot;
  int32_t *match_pos_out;    // [B][Hq] or null
  double rope_w[kHeadDim / 2];
};

enum { MODE_DECODE = 0, MODE_FULL = 1 };

struct AttendParams {
  int mode;
  int check_len;             // flag lengths outside [1, capacity] (MAC_DEV_BAD_SEQ_LEN)
  int B, Hq, Hkv, d, K, r;
  const int32_t *len;        // [B]: m (decode/full) or p - r (seeding)
  int64_t max_len;           // lengths above min(capacity, max_context) are rejected
  KvView kv;
  const float *q_rot;        // [B][Hq][d]
  const int2 *head_info;     // decode: [B][Hq]
  const int32_t *unit_s;     // decode: [B*Hkv]
  const float *ring_o;       // decode: cached summaries [B][Hq][K][d]
  const float *ring_lse;     // decode: [B][Hq][K]
  float *as_o;               // decode: AS_{1:m-r} [B][Hq][d] (may be null)
  float *as_lse;             // decode: [B][Hq] (may be null)
  float *out;                // [B][Hq][d]
  float *out_lse;            // [B][Hq] or null
  int32_t *ctl;
  int32_t *unit_done;
  float *partials;
};

struct RopeParams {
  int B, Hq, d, r, rope_mode, n_seed, seed_index;
  float q_scale;
  const void *q;             // full: [B][Hq][d]; seed: [B][Hq][n_seed][d]
  const int32_t *pos_base;   // [B]
  int pos_add;               // position = pos_base[b] + pos_add
  float *q_rot;
  int32_t *seed_pos;         // seed only: position, or 0 when < 1
  int32_t *seed_len;         // seed only: p - r
  int32_t *ctl;
  double rope_w[kHeadDim / 2];
};

struct AppendParams {
  int B, Hq, d, K, seed_index, n_seed;
  const int32_t *pos;        // [B]: position to append
  int64_t capacity;          // max valid position
  const void *q_src;         // decode: stage_q [B][Hq][d]; seed: q_seed [B][Hq][n_seed][d]
  const float *src_o;        // [B][Hq][d]
  const float *src_lse;      // [B][Hq]
  int32_t *ring_pos;
  void *ring_q;
  float *ring_o;
  float *ring_lse;
};

// ---------------------------------------------------------------------------
// launchers (defined in the .cu files)
// ---------------------------------------------------------------------------
cudaError_t launch_match(const MatchParams &p, int dtype, cudaStream_t s);
cudaError_t launch_rope(const RopeParams &p, int dtype, cudaStream_t s);
cudaError_t launch_append(const AppendParams &p, int dtype, cudaStream_t s);

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
#ifdef __CUDACC__

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for a phase of an mbarrier, giving up after ~2^31 clock cycles (about a
// second); returns false (and the caller reports MAC_DEV_WAIT_TIMEOUT) if the
// phase never completed.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > (1LL << 31)) return false;
  }
  return true;
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 1-D bulk copy (TMA) global -> shared, completion counted in bytes on bar.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// bf16 pair in a 32-bit word -> two floats (element 2i is the low half).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void set_status(int32_t *ctl, int bits) {
  atomicOr(reinterpret_cast<int *>(ctl), bits);
}

// Total order used by every argmin of the match: smaller distance first,
// equal distances prefer the more recent position.
__device__ __forceinline__ bool better(float d_a, int p_a, float d_b, int p_b) {
  return d_a < d_b || (d_a == d_b && p_a > p_b);
}

// Query rotation for one 2x2 block: angle (pos-1) w computed in fp64 and
// reduced modulo 2 pi with a two-part constant (Cody-Waite additive
// reduction), so positions up to 2^31 keep ~1e-7 rad accuracy; the sine and
// cosine of the reduced angle are taken in fp32.
__device__ __forceinline__ void rope_angle(int64_t pos, double w, float *c, float *s) {
  const double kTwoPiHi = 6.283185307179586;      // nearest double to 2 pi
  const double kTwoPiLo = 2.4492935982947064e-16; // 2 pi - kTwoPiHi
  double th = (double)(pos - 1) * w;
  double k = rint(th * (1.0 / 6.283185307179586));
  double rr = fma(-k, kTwoPiHi, th);
  rr = fma(-k, kTwoPiLo, rr);
  sincosf((float)rr, s, c);
}

template <typename T>
__device__ __forceinline__ float elem_f32(const void *base, int64_t i);
template <>
__device__ __forceinline__ float elem_f32<uint16_t>(const void *base, int64_t i) {
  return __uint_as_float((uint32_t)(reinterpret_cast<const uint16_t *>(base)[i]) << 16);
}
template <>
__device__ __forceinline__ float elem_f32<float>(const void *base, int64_t i) {
  return reinterpret_cast<const float *>(base)[i];
}

// q_rot[pair j] = R(pos) q~ scaled by `scale`, for the head whose pre-RoPE
// query starts at element `src` of `q` and whose output starts at `dst`.
// Explicitly rounded operations keep the result bitwise identical wherever
// it is computed (the match kernel for decode steps, the RoPE kernel for
// full attention), so a decode miss and a full-attention call see the same
// query.  Returns false for a non-finite input.
template <typename T>
__device__ __forceinline__ bool rope_rotate_pair(const void *q, int64_t src, float *dst, int j,
                                                 int64_t pos, int mode, double w, float scale) {
  const int half = kHeadDim / 2;
  const int ia = (mode == MAC_ROPE_INTERLEAVED) ? 2 * j : j;
  const int ib = (mode == MAC_ROPE_INTERLEAVED) ? 2 * j + 1 : j + half;
  const float a = elem_f32<T>(q, src + ia), b = elem_f32<T>(q, src + ib);
  float ra = a, rb = b;
  if (mode != MAC_ROPE_NONE) {
    float c, s;
    rope_angle(pos, w, &c, &s);
    ra = __fsub_rn(__fmul_rn(a, c), __fmul_rn(b, s));
    rb = __fadd_rn(__fmul_rn(b, c), __fmul_rn(a, s));
  }
  dst[ia] = __fmul_rn(ra, scale);
  dst[ib] = __fmul_rn(rb, scale);
  return isfinite(a) && isfinite(b);
}

#endif  // __CUDACC__

}  // namespace mac
