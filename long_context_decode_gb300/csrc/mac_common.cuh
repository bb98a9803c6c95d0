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
constexpr int kConsumers = 256;         // span kernel: consumer threads per CTA (8 warps) ...
constexpr int kThreads = kConsumers + 32;  // ... plus one producer warp
constexpr int kWarps = kConsumers / 32;  // consumer warps
constexpr int kStages = 4;              // stage buffers in the span kernel's TMA ring
constexpr int kStageBytes = 32768;      // bytes per stage (K+V tile, or ring rows)
constexpr int kPartStride = kHeadDim + 4;  // floats per (piece, head) partial: o[d], m, l, 0, 0
constexpr int kMaxUnits = 1024;         // B * Hkv
constexpr int kMaxHeads = 4096;         // B * Hq
constexpr int kMaxGrid = 256;           // CTAs of the step grid (one per SM)
constexpr int kGroupCtas = 16;          // CTAs per merge group of a long band
constexpr int kGroups = kMaxGrid / kGroupCtas;
constexpr int kRopeTab = 16;            // requests whose RoPE angles are tabulated per CTA
constexpr int kTracePoints = MAC_TRACE_POINTS;  // timestamps per CTA in a phase trace
constexpr size_t kMaxSmem = 232448;     // dynamic shared memory per CTA (227 KiB)

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// The ring kernel (GQA 8: eight query heads per K/V tile) has its own
// decomposition: every warp feeds and drains a private ring of small stages.
struct TileCounts {
  int nbw, ntt, nsk, nt;
};
namespace ring {
constexpr int kWarps = 8;               // warps per CTA; each feeds and drains its own stage ring
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 3;              // stages in each warp's ring
constexpr int kStageBytes = 8192;       // bytes per stage: a K/V tile, or ring rows
constexpr int kItemStages = 2;          // stages per independent work item (a window tile, a match chunk)
constexpr int kMinSpan = 64;            // fewest long-band tokens worth a CTA

// Tokens of K/V per window tile (one work item): two stages of K and V rows.
__host__ __device__ constexpr int tile_tokens(int elem_bytes) {
  return kItemStages * kStageBytes / (2 * kHeadDim * elem_bytes);
}
// Ring rows per match item.
__host__ __device__ constexpr int item_rows(int elem_bytes) {
  return kItemStages * kStageBytes / (kHeadDim * elem_bytes);
}

// The tiles every unit (request, KV head) attends before the decisions,
// each with its own partial summary: nbw tiles of the band window, cut
// backwards from m - r (it holds every band a hit can need), ntt tiles of
// the tail cut forwards from m - r + 1, and nsk tiles of the front sink.
__host__ __device__ inline TileCounts tile_counts(int K, int r, int64_t max_context, int sink_tokens,
                                                  int elem_bytes) {
  const int T = tile_tokens(elem_bytes);
  const int64_t rr = r < max_context ? r : max_context;
  const int64_t ss = sink_tokens < max_context ? sink_tokens : max_context;
  TileCounts c;
  c.nbw = (K + T - 1) / T;
  c.ntt = (int)((rr + T - 1) / T);
  c.nsk = (int)((ss + T - 1) / T);
  c.nt = c.nbw + c.ntt + c.nsk;
  return c;
}
}  // namespace ring

// ---------------------------------------------------------------------------
// scratch workspace (shared by the kernels of one stream)
// ---------------------------------------------------------------------------
// Span kernel (G <= 4): the tail tokens of all units, laid end to end in
// unit order, are split into one contiguous span per CTA, and so are the
// long bands; a CTA's span meets a few units, each meeting is a piece with
// its own partial summary.  Piece (unit u, CTA c) goes to slot u + c: the
// CTAs meeting a unit form a run that starts at or after the last CTA of
// the previous unit, so the slots of different pieces never coincide and
// B*Hkv + grid - 1 suffice.  A short band is one piece, in band slot u;
// long-band pieces follow at B*Hkv + u + c.  A long band run over more than
// kGroupCtas CTAs is merged in two levels: CTA group k = c / kGroupCtas
// first, into group slot u + k (unique for the same reason), then the
// groups.  The per-head minima and the match's chunk counter live in the
// ring workspace (its match state), double-buffered by the ring's step
// count: step k on a ring combines into copy k & 1 and clears the other for
// step k + 1, so a step needs nothing from the scratch before its match.
//
// Ring kernel (G = 8): window tile t of unit u leaves its partial in part_w
// slot u * nt + t; the long bands are cut over the CTAs as above, the CTA
// meeting unit u leaving its piece in part_c slot u + c, merged per CTA
// group into part_g; part_x holds each CTA's per-warp states while it
// combines them.  Its minima and long-band counts are double-buffered the
// same way.
//
// Everything before `parts` starts at zero and a clean launch leaves it so.
struct ScratchLayout {
  size_t ctl;        // uint32[64]: [0] status word, [2..3] grid-barrier counter (u64),
                     // [4] CTAs of the running launch finished (ring kernel;
                     // the last resets it), [6] decode launch count
  size_t best;       // uint64 [2][B][Hq]: ~(dist bits << 32 | ~pos) of the best candidate, 0 = none
                     // (ring kernel; the span kernel keeps its minima in the ring workspace)
  size_t unit_done;  // uint32 [2][B*Hkv]: pieces (or groups) of the unit finished
  size_t group_done; // uint32 [2][B*Hkv + kGroups]: long-band pieces finished per (unit, CTA group)
  size_t parts;      // first partial (nothing from here on needs clearing)
  // span kernel
  size_t part_a;     // f32 [B*Hkv + kMaxGrid][G][kPartStride]: tail pieces
  size_t part_b;     // f32 [2*B*Hkv + kMaxGrid][G][kPartStride]: band pieces (short
                     // bands at u, long-band pieces at B*Hkv + u + c)
  size_t part_s;     // f32 [B*Hkv][G][kPartStride]: front-sink pieces
  // both
  size_t part_g;     // f32 [B*Hkv + kGroups][G][kPartStride]: merged CTA groups of a long band
  // ring kernel
  size_t part_w;     // f32 [B*Hkv][nt][G][kPartStride]: window, tail and sink tiles
  size_t part_c;     // f32 [B*Hkv + kMaxGrid][G][kPartStride]: long-band CTA pieces
  size_t part_x;     // f32 [kMaxGrid][ring::kWarps][G][kPartStride]: warp states of a CTA piece
  size_t total;
};

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
  float thr2;                // squared match threshold (fp32)
  float q_scale;             // log2(e)/sqrt(d)
  int rope_mode;
  const int32_t *pos_base;
  int pos_add, len_sub;
  int64_t max_len;           // lengths above min(capacity, max_context) are rejected
  KvView kv;
  const void *q;             // query of (b, h) at element (b*Hq + h) * q_stride + q_offset
  int64_t q_stride, q_offset;
  TileCounts tc;             // ring kernel: window tiles per unit (the scratch is sized for these)
  int qslot;                 // ring kernel: the warps' query entries fit in shared memory (0: read from global memory)
  // decode only
  const int32_t *ring_pos;   // [B][K]
  const void *ring_q;        // [B][Hq][K][d]
  const float *ring_o;       // [B][Hq][K][d]
  const float *ring_lse;     // [B][Hq][K]
  void *stage_q;             // [B][Hq][d]: copy of the step's query for the append
  // the ring's match state (span kernel): [0] step count, [2 + k] chunk
  // counter of copy k, then from word 4 the per-head minima u64 [2][B*Hq]
  // (copy k = step count & 1 in use, the other cleared for the next step)
  uint32_t *ring_ctl;
  // fused append (no auxiliary stream): the merges write slot pos mod K of
  // the rings themselves (null: the append kernel does)
  int32_t *app_pos;          // [B][K]
  void *app_q;               // [B][Hq][K][d]
  float *app_o;              // [B][Hq][K][d]
  float *app_lse;            // [B][Hq][K]
  float *as_o;               // [B][Hq][d]: AS_{1:m-r}
  float *as_lse;             // [B][Hq]
  int32_t *match_pos_out;    // [B][Hq] or null
  // outputs
  float *out;                // [B][Hq][d]
  float *out_lse;            // [B][Hq] or null
  // scratch
  uint32_t *ctl;
  unsigned long long *best;  // [2][B*Hq]
  uint32_t *unit_done;       // [2][B*Hkv] (the span kernel uses the first half)
  uint32_t *group_done;      // [2][B*Hkv + kGroups]
  float *part_a, *part_b, *part_s;    // span kernel: tail, band and front-sink pieces
  float *part_w, *part_c, *part_x;    // ring kernel: window tiles, long-band pieces, warp states
  float *part_g;                      // merged CTA groups
  // front sink F: every summary starts at F+1 at the earliest (the reused
  // summaries leave [1, F] out); with sink_piece, [1, min(F, m)] is also
  // attended as output only
  int sink_f, sink_piece;
  unsigned long long *trace;  // optional: [grid][kTracePoints] %globaltimer stamps
  // bounded waits: the budget of every wait on a copy, a flag or another CTA
  // (cycles), and, for the run-out test only, one stage use (>= 0) whose
  // copy is never issued
  long long wait_limit;
  int withhold;
  // host only: launch with programmatic stream serialization (the kernel
  // may start before the previous one on the stream has finished)
  int early_start;
  // RoPE frequency j as a 64-bit fixed-point fraction of a turn per
  // position: round(w_j / (2 pi) * 2^64), w_j = base^(-2j/d)
  unsigned long long rope_f[kHeadDim / 2];
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
// span kernel, G in {1, 2, 4}
cudaError_t launch_step_bf16(const StepParams &p, int grid, cudaStream_t s);
cudaError_t launch_step_f32(const StepParams &p, int grid, cudaStream_t s);
cudaError_t launch_step_bf16_sink(const StepParams &p, int grid, cudaStream_t s);
cudaError_t launch_step_f32_sink(const StepParams &p, int grid, cudaStream_t s);
int step_occupancy_bf16(int G, bool paged, int B, int Hq, int Hkv, int K);
int step_occupancy_f32(int G, bool paged, int B, int Hq, int Hkv, int K);
int step_occupancy_bf16_sink(int G, bool paged, int B, int Hq, int Hkv, int K);
int step_occupancy_f32_sink(int G, bool paged, int B, int Hq, int Hkv, int K);
// the span kernel with the phase trace compiled in (bf16, no front sink)
cudaError_t launch_step_bf16_trace(const StepParams &p, int grid, cudaStream_t s);
// ring kernel, G = 8
namespace ring {
cudaError_t launch_bf16_g8(const StepParams &p, int grid, cudaStream_t s);
cudaError_t launch_f32_g8(const StepParams &p, int grid, cudaStream_t s);
int occupancy_bf16_g8(bool paged, int U, int B);
int occupancy_f32_g8(bool paged, int U, int B);
}  // namespace ring
cudaError_t launch_append(const AppendParams &p, int dtype, cudaStream_t s);
cudaError_t launch_reset(int32_t *ring_pos, int32_t *flags, int B, int K, cudaStream_t s);

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



// Wait for the phase of parity `parity` of an mbarrier, giving up after
// ~2^31 clock cycles (about a second) or as soon as *abort is set; returns
// false when it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile int *abort, long long limit) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort || clock64() - t0 > limit) return false;
  }
  return true;
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

// Same, with an L2 eviction policy (streams read once per step: K/V rows,
// ring rows) so they do not push out what is reused.
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void *src, uint32_t bytes,
                                              uint32_t bar, unsigned long long policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], "
      "%2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}


// Bulk prefetch of global memory into L2 (16-byte aligned, size a
// multiple of 16).
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ unsigned long long l2_evict_first_policy() {
  unsigned long long pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Barrier of the span kernel's consumer threads (all of them).  bar.sync
// counts whole warps, so each warp first reconverges: a lane still inside a
// single-lane region must not be counted as arrived.
__device__ __forceinline__ void consumer_sync() {
  __syncwarp();
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

// Barrier `id` (1..15) of `n` threads (whole warps), after reconverging the
// warp (same reason).
__device__ __forceinline__ void named_sync(int id, int n) {
  __syncwarp();
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// __syncthreads() after reconverging the warp (same reason).
__device__ __forceinline__ void block_sync() {
  __syncwarp();
  __syncthreads();
}

// Programmatic dependent launch: let the next kernel on the stream start
// (its CTAs take SMs as this grid frees them), and wait until the previous
// kernel on the stream has finished with its writes visible (returns at
// once when the launch has no such dependency).
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Orders this thread's earlier shared-memory accesses (generic proxy)
// before its later bulk copies into shared memory (async proxy).
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Hardware approximations (relative error about 2^-22) for normalising
// merged states: the sum of a state is at least 1 (its largest term is
// 2^0), so neither meets a denormal.
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// bf16 pair in a 32-bit word -> two floats (element 2i is the low half).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void set_status(uint32_t *ctl, uint32_t bits) { atomicOr(ctl, bits); }

// 64-bit division, kept out of line: the inlined routine is long and only
// the rare large-size paths need it.
__device__ __noinline__ static long long div_s64(long long a, long long b) { return a / b; }

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Query rotation angle of one 2x2 block, (pos-1) w_j modulo 2 pi, from the
// frequency as a 64-bit fixed-point fraction of a turn (f = w_j / 2pi * 2^64):
// the product (pos-1) f taken modulo 2^64 is the angle's fraction of a turn,
// exact up to the rounding of f (relative 2^-53), read as a signed value so
// the angle lands in [-pi, pi).  Its sine and cosine come from the hardware
// approximations (absolute error about 4e-7 on [-pi, pi]).  All integer and
// fp32 arithmetic: GB300's fp64 rate is a small fraction of its fp32 rate.
__device__ __forceinline__ void rope_angle(int64_t pos, unsigned long long f, float *c, float *s) {
  const unsigned long long turn = (unsigned long long)(pos - 1) * f;
  const float a = (float)(long long)turn * 3.4061215800865545e-19f;  // 2 pi / 2^64
  __sincosf(a, s, c);
}

// b - c for a bf16 b (its bits) and an f32 c, rounded once to f32 (the
// mixed-precision subtraction of sm_100 and later)
__device__ __forceinline__ float bf16_minus_f32(uint16_t b, float c) {
  float d;
  asm("sub.rn.f32.bf16 %0, %1, %2;" : "=f"(d) : "h"(b), "f"(c));
  return d;
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

#endif  // __CUDACC__

}  // namespace mac
