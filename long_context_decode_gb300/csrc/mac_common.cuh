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
constexpr int kHeadDim = 128;           // supported head dimension
constexpr int kThreads = 256;           // threads per CTA (8 warps; thread 0 also issues the copies)
constexpr int kConsumers = kThreads;
constexpr int kWarps = kThreads / 32;
constexpr int kStages = 5;              // stage buffers in the TMA ring
constexpr int kStageBytes = 32768;      // bytes per stage (K+V tile, or ring rows)
constexpr int kTailChunk = 128;         // tokens per tail chunk (the last r positions)
constexpr int kBandChunkMin = 128;      // band chunk size grows from here ...
constexpr int kBandChunkMax = 1024;     // ... up to here, so that a unit has at most
constexpr int kBandChunksTarget = 128;  //     kBandChunksTarget band chunks when possible
constexpr int kPartStride = kHeadDim + 4;  // floats per (item, head) partial: o[d], m, l, 0, 0
constexpr int kMaxUnits = 1024;         // B * Hkv
constexpr int kMaxHeads = 4096;         // B * Hq
constexpr int kTracePoints = 8;         // timestamps per CTA in a phase trace

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------------------
// scratch workspace (shared by the kernels of one stream)
// ---------------------------------------------------------------------------
struct ScratchLayout {
  size_t ctl;        // uint32[64]: [0] status word, [1] grid-barrier counter
  size_t best;       // uint64 [B][Hq]: ~(dist bits << 32 | ~pos) of the best candidate, 0 = none
  size_t match_cnt;  // int32 [B*Hkv]: CTAs whose match slice covered the unit and finished
  size_t head_info;  // int2 [B][Hq]: {matched position or -1, first fresh token lo}
  size_t unit_s;     // int32 [B*Hkv]: first token any head of the unit reads
  size_t tail_part;  // f32 [B*Hkv][n_tail][G][kPartStride]: tail chunk partials
  size_t partials;   // f32 [max_items][G][kPartStride]: band chunk partials
  size_t total;
  int64_t max_items;
};

// ---------------------------------------------------------------------------
// per-(request, kv-head) chunk plan
// ---------------------------------------------------------------------------
// The fresh range of a unit is [s, m] (s = first token any head of the group
// needs).  It is cut at m-r: band chunks cover [s, m-r] and end on m-r,
// tail chunks (tail_range) cover [m-r+1, m] in kTailChunk pieces aligned on
// m-r.  Every chunk lies wholly on one side of m-r, so per head the band
// chunks (plus the cached summary) give the rectified summary AS_{1:m-r} and
// the tail chunks complete the output ([MAC] K2/K3).  The same plan with
// s = 1 is the exact full attention, which makes a miss bitwise equal to it.
struct BandPlan {
  int64_t m, s;
  int32_t cb, nb;  // chunk size and number of band chunks
};

__host__ __device__ inline BandPlan plan_band(int64_t m, int64_t s, int r) {
  BandPlan u;
  u.m = m;
  u.s = s;
  const int64_t band_len = (m - r) - s + 1;
  u.cb = kBandChunkMin;
  u.nb = 0;
  if (m >= 1 && band_len > 0) {
    while (u.cb < kBandChunkMax && (band_len + u.cb - 1) / u.cb > kBandChunksTarget) u.cb <<= 1;
    u.nb = (int32_t)((band_len + u.cb - 1) / u.cb);
  }
  return u;
}

// Token range [lo, hi] of band chunk i of the unit.
__host__ __device__ inline void band_range(const BandPlan &u, int r, int i, int64_t *lo,
                                           int64_t *hi) {
  const int64_t top = (u.m - r) - (int64_t)(u.nb - 1 - i) * u.cb;
  const int64_t bot = top - u.cb + 1;
  *lo = bot > u.s ? bot : u.s;
  *hi = top;
}

// Worst-case band chunks per unit for contexts up to max_context.
__host__ inline int64_t max_band_items_per_unit(int64_t max_context) {
  int64_t nb = kBandChunksTarget;
  int64_t by_max = (max_context + kBandChunkMax - 1) / kBandChunkMax;
  if (by_max > nb) nb = by_max;
  return nb + 1;
}

// Number of tail chunks of a unit (the last r tokens in kTailChunk pieces).
__host__ __device__ inline int n_tail_chunks(int r) { return (r + kTailChunk - 1) / kTailChunk; }

// Token range of tail chunk j of a request at length m: the chunks are
// aligned on m-r and clipped to [1, m] (empty when lo > hi).  They do not
// depend on the match: every head's band start lies at or before m-r+1.
__host__ __device__ inline void tail_range(int64_t m, int r, int j, int64_t *lo, int64_t *hi) {
  const int64_t base = m - r + 1 + (int64_t)j * kTailChunk;
  *lo = base > 1 ? base : 1;
  const int64_t top = base + kTailChunk - 1;
  *hi = top < m ? top : m;
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

enum { MODE_DECODE = 0, MODE_FULL = 1 };

// One launch of the step kernel.  Positions and lengths of request b:
//   pos = pos_base[b] + pos_add      (the query's position: RoPE angle pos-1)
//   m   = pos - len_sub              (attention over [1, m]; decode/full: 0)
struct StepParams {
  int mode;
  int check_len;             // flag lengths outside [1, max_len] (MAC_DEV_BAD_SEQ_LEN)
  int B, Hq, Hkv, G, K, r, min_context;
  int n_tail;                // tail chunks per unit, n_tail_chunks(r)
  float thr2;                // squared match threshold (fp32)
  float q_scale;             // log2(e)/sqrt(d)
  int rope_mode;
  const int32_t *pos_base;
  int pos_add, len_sub;
  int64_t max_len;           // lengths above min(capacity, max_context) are rejected
  KvView kv;
  const void *q;             // query of (b, h) at element (b*Hq + h) * q_stride + q_offset
  int64_t q_stride, q_offset;
  // decode only
  const int32_t *ring_pos;   // [B][K]
  const void *ring_q;        // [B][Hq][K][d]
  const float *ring_o;       // [B][Hq][K][d]
  const float *ring_lse;     // [B][Hq][K]
  void *stage_q;             // [B][Hq][d]: copy of the step's query for the append
  float *as_o;               // [B][Hq][d]: AS_{1:m-r}
  float *as_lse;             // [B][Hq]
  int32_t *match_pos_out;    // [B][Hq] or null
  // outputs
  float *out;                // [B][Hq][d]
  float *out_lse;            // [B][Hq] or null
  // scratch
  uint32_t *ctl;
  unsigned long long *best;
  int32_t *match_cnt;
  int2 *head_info;
  int32_t *unit_s;
  float *tail_part;
  float *partials;
  unsigned long long *trace;  // optional: [grid][kTracePoints] %globaltimer stamps
  double rope_w[kHeadDim / 2];
};

struct AppendParams {
  int B, Hq, K;
  const int32_t *pos_base;   // position appended for request b: pos_base[b] + pos_add
  int pos_add;
  int64_t capacity;          // max valid position
  const void *q_src;         // query of (b, h) at element (b*Hq + h) * q_stride + q_offset
  int64_t q_stride, q_offset;
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
cudaError_t launch_step_bf16(const StepParams &p, int grid, cudaStream_t s);
cudaError_t launch_step_f32(const StepParams &p, int grid, cudaStream_t s);
int step_occupancy_bf16(int G, bool paged, int n_units);
int step_occupancy_f32(int G, bool paged, int n_units);
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

// Non-blocking test of the phase of parity `parity`.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of parity `parity` of an mbarrier, giving up after
// ~2^31 clock cycles (about a second) or as soon as *abort is set; returns
// false when it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile int *abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort || clock64() - t0 > (1LL << 31)) return false;
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

// Barrier of the CTA's consumer threads (all of them).
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// bf16 pair in a 32-bit word -> two floats (element 2i is the low half).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void set_status(uint32_t *ctl, uint32_t bits) { atomicOr(ctl, bits); }

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
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

// dst[pair j] = R(pos) q~ scaled by `scale`, for the head whose pre-RoPE
// query starts at element `src` of `q` and whose output starts at `dst`.
// Explicitly rounded operations keep the result bitwise identical wherever
// it is computed, so a decode miss and a full-attention call see the same
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
