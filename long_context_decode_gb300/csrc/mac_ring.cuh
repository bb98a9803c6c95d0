// mac_ring.cuh -- the decode step for GQA groups of eight query heads: one
// persistent kernel per step (cooperative launch, one CTA of eight warps per
// SM).  Every warp feeds and drains its own ring
// of shared-memory stages: its first lane issues the 1-D bulk (TMA) copies a
// few stages ahead of the stage the warp is working on, so the streaming
// phases hold no CTA barrier.
//
//   Phase A -- work that needs no decision, as independent 16 KB items dealt
//   round-robin to all warps of the grid:
//     * match items ([MAC] "Match (2)"/"Match (3)", K1): 64 rows of one
//       head's pre-RoPE query ring.  Eight lanes share a row; each sums
//       (a-b)^2 of its 16 elements (a-b of two bf16 values is exact in fp32)
//       as two pairwise trees, one per half of the dims; the eight lanes
//       finish each half's tree with shuffles and the distance is the sum of
//       the halves: at most 8 roundings of non-negative terms.  The pages'
//       expansion |a|^2+|b|^2-2a.b cancels badly for close pairs and is not
//       used.  The warp's best (distance, position) joins the head's minimum
//       through a 64-bit atomic max of a packed key, a total order (smaller
//       distance, then the more recent position), so the result does not
//       depend on scheduling.
//     * window tiles ([MAC] "Complete", K2): every unit (request, KV head)
//       attends the last K + r tokens before the decisions exist, as tiles of
//       32 tokens cut backwards from m - r (the band window: a hit at
//       p >= m - K needs the band [p - r + 1, m - r], which lies in it) and
//       forwards from m - r + 1 (the tail), plus the front sink when there is
//       one.  Each tile leaves one partial summary per head (running max,
//       sum, weighted values; base-2 log domain); a GQA group loads each K/V
//       tile once for its G query heads.
//   Grid barrier; the minima become decisions ([MAC] K1: hit iff the
//   smallest squared distance is strictly below thr^2).
//   Phase B:
//     * hits: the band of a hit at p starts at lo = p - r + 1, inside one
//       window tile; the unit's owner CTA re-attends that tile from lo on
//       for the head (its later tiles are whole), then merges the cached
//       rectified summary of [1, p - r], the boundary piece and the band
//       tiles into AS_{1:m-r}, and that with the tail into the output
//       ([MAC] "Decomposable attention", "Amend"; [ACSP] log-sum-exp merge).
//     * misses ([MAC] "Match (1)": exact attention): the rest of [1, m]
//       before the window (the long band) of every unit with a missing head,
//       laid end to end and cut into one span per CTA; the eight warps of a
//       CTA take its stages round-robin and combine their states per unit;
//       the CTAs' pieces are merged per group of kGroupCtas CTAs by the last
//       to finish, and the owner merges the groups with the window tiles.
//   Full attention (and ring seeding) run the same kernel with every head
//   missing and no match, so a decode step whose heads all miss is bitwise
//   equal to full attention.
//
// Every wait is bounded and reports MAC_DEV_WAIT_TIMEOUT instead of hanging.
#pragma once

#include "mac_common.cuh"

namespace mac {
namespace ring {

// Candidate key: smaller distance first, then the more recent position.
// Stored inverted so that an atomic max keeps the best one and 0 means
// "no candidate" (distances are >= 0, whose float bits order like unsigned).
__device__ __forceinline__ unsigned long long pack_best(float d, int pos) {
  const unsigned long long key = ((unsigned long long)__float_as_uint(d) << 32) |
                                 (unsigned long long)(0xFFFFFFFFu - (uint32_t)pos);
  return ~key;
}

__device__ __forceinline__ bool better(float d_a, int p_a, float d_b, int p_b) {
  return d_a < d_b || (d_a == d_b && p_a > p_b);
}

__device__ __forceinline__ unsigned long long atom_add_release_u64(unsigned long long *p, unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.add.release.gpu.global.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
  return old;
}

// A count of finished pieces: release of the partials the calling CTA wrote
// before its barrier, acquire of those the earlier counts released.
__device__ __forceinline__ uint32_t atom_add_acq_rel_u32(uint32_t *p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// The partial of an empty merge entry: zero sum and output.
static __device__ __align__(16) float g_zero_partial[kPartStride];

// 16 bytes of elements -> pairs of consecutive elements as float2.
template <typename T>
__device__ __forceinline__ void unpack16x2(const uint4 &u, float2 *f);
template <>
__device__ __forceinline__ void unpack16x2<uint16_t>(const uint4 &u, float2 *f) {
  f[0] = make_float2(bf16_lo(u.x), bf16_hi(u.x));
  f[1] = make_float2(bf16_lo(u.y), bf16_hi(u.y));
  f[2] = make_float2(bf16_lo(u.z), bf16_hi(u.z));
  f[3] = make_float2(bf16_lo(u.w), bf16_hi(u.w));
}
template <>
__device__ __forceinline__ void unpack16x2<float>(const uint4 &u, float2 *f) {
  f[0] = make_float2(__uint_as_float(u.x), __uint_as_float(u.y));
  f[1] = make_float2(__uint_as_float(u.z), __uint_as_float(u.w));
}

constexpr int ilog2c(int x) { return x <= 1 ? 0 : 1 + ilog2c(x >> 1); }

// Running maxima start here (finite, so that empty states never produce
// inf - inf) and are raised only when a score exceeds them by kLazy (base-2
// log units): the accumulators then stay within 2^kLazy of the true scale.
constexpr float kMInit = -1e30f;
constexpr float kLazy = 8.f;
constexpr unsigned kFull = 0xffffffffu;
constexpr int32_t kNoPage = (int32_t)0x80000000;

template <typename T, int G, bool PAGED>
struct Step {
  static constexpr int kES = (int)sizeof(T);
  static constexpr int kRow = kHeadDim * kES;                 // bytes of a K, V or ring row
  static constexpr int kStTok = kStageBytes / (2 * kRow);     // K/V tokens per stage: 16 / 8
  static constexpr int kTT = kStTok * kItemStages;            // tokens per window tile: 32 / 16
  static constexpr int kStRows = kStageBytes / kRow;          // ring rows per stage: 32 / 16
  static constexpr int kIR = kStRows * kItemStages;           // ring rows per match item
  static constexpr int kPer = 16 / kES;                       // elements per 16-byte load
  // match: 8 lanes per row, lane `sub` owns dims [8 sub, 8 sub + 8) of
  // each half of the row; kMRG rows per lane group of a stage
  static constexpr int kHalfLoads = 8 / kPer;                 // 16-byte loads per half: 1 / 2
  static constexpr int kMRG = kStRows / 4;                    // 8 / 4
  static constexpr int kLogMRG = ilog2c(kMRG);
  // attention: a half-warp per token, lane `sub` (0..15) owns dims
  // [8 sub, 8 sub + 8) of the query and the weighted values; kATPG tokens
  // per half-warp per pass, one score per lane after a reduce-scatter
  static constexpr int kATPG = G <= 4 ? 4 : 2;
  static constexpr int kPassTok = 2 * kATPG;
  static constexpr int kPasses = kStTok / kPassTok;
  static constexpr int kAV = kATPG * G;
  static constexpr int kAScat = ilog2c(kAV);
  static constexpr int kAPlain = 4 - kAScat;
  static constexpr int kLogG = ilog2c(G);
  static constexpr int kLogATPG = ilog2c(kATPG);
  static constexpr int kAPairs = 4;                           // float2 per lane and head
  static constexpr int kALoads = 8 * kES / 16;                // 16-byte loads per lane and row
  // merges: kWPH warps per head, each owning kDW dims (kDL per lane)
  static constexpr int kWPH = kWarps / G;
  static constexpr int kDW = kHeadDim / kWPH;
  static constexpr int kDL = kDW >= 32 ? kDW / 32 : 1;
  static constexpr int kLanes = kDW / kDL;
  static_assert(kAV <= 16 && kAV >= 2, "one score per lane of a half-warp at most");
  static_assert(kPasses >= 1 && kPasses * kPassTok == kStTok, "passes per stage");
  static_assert(kStTok <= 16, "a stage meets at most two 16-token pages");

  // dynamic shared memory layout
  static constexpr size_t kOffBar = (size_t)kWarps * kStages * kStageBytes;
  static constexpr size_t kOffMask = kOffBar + 8 * kWarps * kStages;      // int [kWarps][kStages]
  static constexpr size_t kOffBd = kOffMask + 4 * kWarps * kStages;       // f32 [kWarps][kPartStride]
  static constexpr size_t kOffUnits = kOffBd + 4 * (size_t)kWarps * kPartStride;
  static_assert(kOffBar % 8 == 0 && kOffBd % 16 == 0 && kOffUnits % 16 == 0, "alignment");
  // + the long-band offsets (int64 [U + 1]) and unit lengths (int32 [U]),
  // then, for at most kRopeTab requests, the cos and sin of every request's
  // query rotation angles (float2 [B][d/2])
  static constexpr int kRopeTab = 16;
  __host__ __device__ static size_t off_rope(int U) {
    return (kOffUnits + 8 * (size_t)(U + 1) + 4 * (size_t)U + 15) / 16 * 16;
  }
  // + each stage's ring positions (a match stage's rows: int32 [kStRows]),
  // then (when there is room) each warp's two query entries: a unit's G
  // query rows or a head's, copied with the first stage of an item whose
  // query differs from the item before
  static constexpr int kPosBytes = kStRows * 4;
  static constexpr int kQE = G * kRow;
  static constexpr int kQBuf = kWarps * 2 * kQE;
  __host__ __device__ static size_t off_pside(int U, int B) {
    return off_rope(U) + (B <= kRopeTab ? 8 * (size_t)B * (kHeadDim / 2) : 0);
  }
  __host__ __device__ static size_t off_qbuf(int U, int B) {
    return off_pside(U, B) + (size_t)kWarps * kStages * kPosBytes;
  }
  __host__ __device__ static size_t smem_bytes(int U, int B) { return off_qbuf(U, B); }

  struct Smem {
    uint8_t *stage;     // [kWarps][kStages][kStageBytes]
    uint64_t *full;     // [kWarps][kStages]: the stage's copy has landed
    int *rows;          // [kWarps][kStages]: rows of the stage that were copied (bit mask)
    float *bd;          // [kWarps][kPartStride]: boundary pieces of a batch of owned heads
    int64_t *off;       // [U + 1]: long-band offsets (units end to end)
    int32_t *um;        // [U]: the unit's length m (0: not a valid length)
    long long *scan;    // [kWarps]
    volatile int *abort;
    int64_t *ntok;      // long-band tokens in all
    int *Pl;            // CTAs the long bands are cut over
    unsigned long long *best, *best_next;
    volatile uint32_t *flag;
    int *dec;           // [kOwnMax]: decisions of the heads this CTA owns
    uint32_t *unit_done, *group_done;            // this launch's long-band counts
    uint32_t *unit_done_next, *group_done_next;  // cleared here for the next launch
    float2 *rope;       // [B][d/2] cos, sin of the query angles (B <= kRopeTab), or null
    uint8_t *pside;     // [kWarps][kStages][kPosBytes]: ring positions of match stages
    uint8_t *qbuf;      // [kWarps][2][kQE]: query entries, or null (queries read from global memory)
  };

  // One warp's ring: stage uses are numbered; use n sits in stage n % kStages.
  struct Ring {
    uint8_t *buf;       // this warp's kStages stages
    uint32_t bar0;      // shared address of its first full barrier
    int *rows;
    uint8_t *pside;     // this warp's stage position buffers
    uint8_t *qbuf;      // this warp's two query entries (or null)
    uint32_t issued, used;
  };

  // What one stage use holds: K/V rows [a, a + cnt) of unit u (kind 1), or
  // ring rows [a, a + cnt) of head u (kind 2); kind 0: nothing; -1: the end.
  struct Desc {
    int kind = -1, u = 0, a = 0, cnt = 0;
    int qe = -1;   // >= 0: also copy the item's query (unit u's G rows; head u's for kind 2) into entry qe
    int pc = 0;    // a match stage whose ring positions come into its position buffer
    int keep = 0;  // K/V rows kept in L2 (read again by a boundary piece)
  };

  __device__ static int lane_id() { return threadIdx.x & 31; }
  __device__ static int warp_id() { return threadIdx.x >> 5; }

  // ---------------------------------------------------------------------
  // unit geometry
  // ---------------------------------------------------------------------
  // lb: the first token a summary covers (F + 1; 1 for full attention).
  __device__ static int lb(const StepParams &p) { return p.sink_f + 1; }
  __device__ static bool len_ok(const StepParams &p, int64_t m) { return m >= 1 && m <= p.max_len; }
  // window start: the earliest band start a hit can have
  __device__ static int win_start(const StepParams &p, int m) { return max(lb(p), m - p.r - p.K + 1); }
  __device__ static int tail_start(const StepParams &p, int m) { return max(lb(p), m - p.r + 1); }
  // Tile t of a unit of length m (0 when invalid): tokens [*lo, *hi] (empty when *lo > *hi).
  __device__ static void tile_range(const StepParams &p, int m, int t, int *lo, int *hi) {
    *lo = 1;
    *hi = 0;
    if (m <= 0) return;
    if (t < p.tc.nbw) {
      const int h = m - p.r - kTT * t;
      *hi = h;
      *lo = max(win_start(p, m), h - kTT + 1);
    } else if (t < p.tc.nbw + p.tc.ntt) {
      const int l = tail_start(p, m) + kTT * (t - p.tc.nbw);
      *lo = l;
      *hi = min(m, l + kTT - 1);
    } else if (p.sink_piece) {
      const int l = 1 + kTT * (t - p.tc.nbw - p.tc.ntt);
      *lo = l;
      *hi = min(min(p.sink_f, m), l + kTT - 1);
    }
  }
  // the request's query position (RoPE angle pos - 1)
  __device__ static int64_t qpos(const StepParams &p, int b) { return (int64_t)p.pos_base[b] + p.pos_add; }

  // ---------------------------------------------------------------------
  // copies
  // ---------------------------------------------------------------------
  __device__ static uint8_t *stage_buf(const Ring &R, uint32_t n) {
    return R.buf + (size_t)(n % kStages) * kStageBytes;
  }
  __device__ static uint32_t stage_bar(const Ring &R, uint32_t n) { return R.bar0 + 8 * (n % kStages); }

  // Page ids of the (at most two) pages a K/V stage meets, loaded ahead of
  // its copy (kNoPage: none).
  __device__ static void load_ids(const StepParams &p, const Desc &d, int32_t (&id)[2]) {
    id[0] = id[1] = kNoPage;
    if (!PAGED || d.kind != 1 || d.cnt <= 0 || lane_id() != 0 || d.u < 0 || d.u >= p.B * p.Hkv) return;
    const int b = d.u / p.Hkv;
    const int s0 = (d.a - 1) >> 4, s1 = (d.a + d.cnt - 2) >> 4;
    const int32_t *row = p.kv.page_table + (int64_t)b * p.kv.max_pages;
    if (s0 >= 0 && s0 < p.kv.max_pages) id[0] = __ldg(row + s0);
    if (s1 != s0 && s1 < p.kv.max_pages) id[1] = __ldg(row + s1);
  }

  // The query copy that rides with a stage: bytes, and its issue.
  __device__ static uint32_t query_bytes(const Desc &d, const Ring &R) {
    return d.qe >= 0 && R.qbuf ? (d.kind == 2 ? (uint32_t)kRow : (uint32_t)kQE) : 0u;
  }
  __device__ static void issue_query(const StepParams &p, const Ring &R, const Desc &d, uint32_t bar) {
    uint8_t *dst = R.qbuf + (size_t)d.qe * kQE;
    const uint8_t *q = (const uint8_t *)p.q;
    if (d.kind == 2) {
      bulk_g2s(smem_addr(dst), q + ((int64_t)d.u * p.q_stride + p.q_offset) * kES, kRow, bar);
      return;
    }
    const int b = d.u / p.Hkv, g = d.u - b * p.Hkv;
    const int64_t bh0 = (int64_t)b * p.Hq + g * G;
    if (p.q_stride == kHeadDim && p.q_offset == 0) {  // the unit's G rows are contiguous
      bulk_g2s(smem_addr(dst), q + bh0 * kRow, kQE, bar);
    } else {
      for (int hh = 0; hh < G; ++hh)
        bulk_g2s(smem_addr(dst + hh * kRow), q + ((bh0 + hh) * p.q_stride + p.q_offset) * kES, kRow, bar);
    }
  }

  // Lane 0: the copies of the next stage use (every lane calls it).
  __device__ static void issue(const StepParams &p, Ring &R, const Desc &d, const int32_t (&id)[2]) {
    const uint32_t n = R.issued++;
    if (lane_id() != 0 || (int)n == p.withhold) return;  // the run-out test's use is never copied
    uint8_t *buf = stage_buf(R, n);
    const uint32_t bar = stage_bar(R, n);
    int *rows = R.rows + n % kStages;
    const uint32_t qb = query_bytes(d, R);
    if (d.kind == 2) {  // ring rows of head d.u (and their positions)
      const uint32_t bytes = (uint32_t)d.cnt * kRow;
      *rows = (1 << d.cnt) - 1;
      mbar_expect_tx(bar, bytes + qb + (d.pc ? 4u * d.cnt : 0u));
      if (qb) issue_query(p, R, d, bar);
      if (d.pc)
        bulk_g2s(smem_addr(R.pside + (size_t)(n % kStages) * kPosBytes),
                 p.ring_pos + (int64_t)(d.u / p.Hq) * p.K + d.a, 4u * d.cnt, bar);
      bulk_g2s_hint(smem_addr(buf), (const uint8_t *)p.ring_q + ((size_t)d.u * p.K + d.a) * kRow, bytes, bar,
                    l2_evict_first_policy());
      return;
    }
    const int g = d.u % p.Hkv;
    int msk = 0;
    uint32_t bytes = 0;
    bool ok = d.kind == 1 && d.cnt > 0;
    if (ok && !PAGED && (d.a < 1 || d.a + d.cnt - 1 > p.kv.capacity || d.u >= p.B * p.Hkv)) {
      set_status(p.ctl, MAC_DEV_BAD_COPY);
      ok = false;
    }
    const int n0 = ok ? min(d.cnt, 16 - ((d.a - 1) & 15)) : 0;  // rows of the first page (paged)
    if (ok && !PAGED) {
      msk = (1 << d.cnt) - 1;
      bytes = 2u * (uint32_t)d.cnt * kRow;
    } else if (ok) {
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        const int cnt = s ? d.cnt - n0 : n0;
        if (cnt <= 0 || id[s] == kNoPage) continue;
        if (id[s] < 0 || id[s] >= p.kv.n_pages) {
          set_status(p.ctl, MAC_DEV_BAD_PAGE);
          continue;
        }
        msk |= s ? ((1 << d.cnt) - 1) & ~((1 << n0) - 1) : (1 << n0) - 1;
        bytes += 2u * (uint32_t)cnt * kRow;
      }
    }
    *rows = msk;
    if (bytes + qb == 0) {
      mbar_arrive(bar);
      return;
    }
    mbar_expect_tx(bar, bytes + qb);
    if (qb) issue_query(p, R, d, bar);
    if (bytes == 0) return;
    if (!PAGED) {
      const size_t off = ((size_t)d.u * (size_t)p.kv.capacity + (size_t)(d.a - 1)) * kRow;
      const uint32_t nb = (uint32_t)d.cnt * kRow;
      if (d.keep) {
        bulk_g2s(smem_addr(buf), (const uint8_t *)p.kv.k + off, nb, bar);
        bulk_g2s(smem_addr(buf + kStageBytes / 2), (const uint8_t *)p.kv.v + off, nb, bar);
      } else {
        const unsigned long long pol = l2_evict_first_policy();
        bulk_g2s_hint(smem_addr(buf), (const uint8_t *)p.kv.k + off, nb, bar, pol);
        bulk_g2s_hint(smem_addr(buf + kStageBytes / 2), (const uint8_t *)p.kv.v + off, nb, bar, pol);
      }
      return;
    }
    const unsigned long long pol = l2_evict_first_policy();
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int cnt = s ? d.cnt - n0 : n0;
      if (cnt <= 0 || !((msk >> (s ? n0 : 0)) & 1)) continue;
      const int t0 = s ? d.a + n0 : d.a;  // first token of the segment
      const size_t off = (((size_t)id[s] * p.Hkv + g) * 16 + (size_t)((t0 - 1) & 15)) * kRow;
      uint8_t *dst = buf + (size_t)(t0 - d.a) * kRow;
      bulk_g2s_hint(smem_addr(dst), (const uint8_t *)p.kv.k + off, (uint32_t)cnt * kRow, bar, pol);
      bulk_g2s_hint(smem_addr(dst + kStageBytes / 2), (const uint8_t *)p.kv.v + off, (uint32_t)cnt * kRow, bar,
                    pol);
    }
  }

  // Wait for stage use n to land (bounded).
  __device__ static bool wait_stage(const StepParams &p, const Smem &S, const Ring &R, uint32_t n) {
    const bool ok = mbar_wait_bounded(stage_bar(R, n), (n / kStages) & 1u, S.abort, p.wait_limit);
    if (!ok && !*S.abort) {
      set_status(p.ctl, MAC_DEV_WAIT_TIMEOUT);
      *S.abort = 1;
    }
    return ok;
  }
  // The warp is done reading its oldest stage: its buffer may be refilled.
  __device__ static void done_with_stage() {
    __syncwarp();
    fence_proxy_async();
  }
  // Before the CTA exits: the copies this warp issued have landed (bounded).
  __device__ static void drain(const StepParams &p, const Ring &R) {
    // a copy lands within microseconds; the bound only guards a stage whose
    // phase a withheld use shifted (the run-out test)
    const long long lim = p.wait_limit < (1LL << 30) ? (p.wait_limit > (1LL << 20) ? p.wait_limit : (1LL << 20))
                                                     : (1LL << 30);
    for (uint32_t n = R.used; n < R.issued; ++n) {
      if ((int)n == p.withhold) continue;
      const long long t0 = clock64();
      while (!mbar_try_wait(stage_bar(R, n), (n / kStages) & 1u) && clock64() - t0 < lim) {
      }
    }
  }

  // ---------------------------------------------------------------------
  // attention of a stage
  // ---------------------------------------------------------------------
  struct Att {
    float2 o[G][kAPairs];
    float mrun[G];
    float m_mine, l_mine;
  };
  __device__ static void att_init(Att &A) {
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      A.mrun[hh] = kMInit;
#pragma unroll
      for (int i = 0; i < kAPairs; ++i) A.o[hh][i] = make_float2(0.f, 0.f);
    }
    A.m_mine = kMInit;
    A.l_mine = 0.f;
  }

  // v[i] (i = token slot * G + head, partial dot products of the lane's 8
  // dims) -> the full dot product of slot sub >> kAPlain: reduce-scatter
  // over the half-warp (xor 8, 4, ...), then plain butterflies for the rest.
  __device__ static float reduce_scores(float (&v)[kAV], int lane) {
#pragma unroll
    for (int lev = 0; lev < kAScat; ++lev) {
      const int off = 8 >> lev;
      const bool up = (lane & off) != 0;
      const int half = kAV >> (lev + 1);
#pragma unroll
      for (int i = 0; i < kAV / 2; ++i) {
        if (i < half) {
          const float send = up ? v[i] : v[i + half];
          const float keep = up ? v[i + half] : v[i];
          v[i] = keep + __shfl_xor_sync(kFull, send, off);
        }
      }
    }
    float s = v[0];
#pragma unroll
    for (int lev = kAScat; lev < 4; ++lev) s += __shfl_xor_sync(kFull, s, 8 >> lev);
    return s;
  }
  // max / sum over the lanes of the half-warp whose score slots hold the
  // same head (the token bits of the slot index)
  __device__ static float head_max(float x) {
#pragma unroll
    for (int b = 0; b < kLogATPG; ++b) x = fmaxf(x, __shfl_xor_sync(kFull, x, 1 << (kAPlain + kLogG + b)));
    return x;
  }
  __device__ static float head_sum(float x) {
#pragma unroll
    for (int b = 0; b < kLogATPG; ++b) x += __shfl_xor_sync(kFull, x, 1 << (kAPlain + kLogG + b));
    return x;
  }

  // One stage: rows 0..kStTok-1 hold tokens a, a+1, ... (K in the first half
  // of the stage, V in the second; `rows` marks the rows actually copied).
  // The lane's score slot counts for its head only within [lo_m, hi_m].
  __device__ static void att_stage(Att &A, const float2 (&q)[G][kAPairs], const uint8_t *buf, int a, int rows,
                                   int lo_m, int hi_m) {
    const int lane = lane_id(), sub = lane & 15, hw = lane >> 4;
    const int idx = sub >> kAPlain, ti = idx / G;
    const uint8_t *kb = buf, *vb = buf + kStageBytes / 2;
#pragma unroll 1
    for (int ps = 0; ps < kPasses; ++ps) {
      float v[kAV];
#pragma unroll
      for (int tt = 0; tt < kATPG; ++tt) {
        const int row = ps * kPassTok + tt * 2 + hw;
        float2 kf[kAPairs];
#pragma unroll
        for (int c = 0; c < kALoads; ++c)
          unpack16x2<T>(*reinterpret_cast<const uint4 *>(kb + row * kRow + sub * 8 * kES + c * 16),
                        kf + c * (kAPairs / kALoads));
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          float2 acc = __fmul2_rn(q[hh][0], kf[0]);
#pragma unroll
          for (int i = 1; i < kAPairs; ++i) acc = __ffma2_rn(q[hh][i], kf[i], acc);
          v[tt * G + hh] = acc.x + acc.y;
        }
      }
      float s = reduce_scores(v, lane);
      const int row_m = ps * kPassTok + ti * 2 + hw, t_m = a + row_m;
      const bool valid = ((rows >> row_m) & 1) && t_m >= lo_m && t_m <= hi_m;
      s = valid ? s : -INFINITY;
      // lazy running max (per half-warp and head): raised only when a score
      // exceeds it by kLazy
      const float mt = head_max(s);
      if (__any_sync(kFull, mt > A.m_mine + kLazy)) {
        const float mn_mine = fmaxf(A.m_mine, mt);
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          const float mn = __shfl_sync(kFull, mn_mine, (lane & 16) | (hh << kAPlain));
          const float f = ex2(A.mrun[hh] - mn);
          const float2 f2 = make_float2(f, f);
#pragma unroll
          for (int i = 0; i < kAPairs; ++i) A.o[hh][i] = __fmul2_rn(A.o[hh][i], f2);
          A.mrun[hh] = mn;
        }
        A.l_mine *= ex2(A.m_mine - mn_mine);
        A.m_mine = mn_mine;
      }
      const float w = ex2(s - A.m_mine);
      A.l_mine += w;
#pragma unroll
      for (int tt = 0; tt < kATPG; ++tt) {
        const int row = ps * kPassTok + tt * 2 + hw;
        uint4 raw[kALoads];
#pragma unroll
        for (int c = 0; c < kALoads; ++c)
          raw[c] = *reinterpret_cast<const uint4 *>(vb + row * kRow + sub * 8 * kES + c * 16);
        // rows not copied hold stale bytes, possibly NaN patterns (0 * NaN is NaN)
        const uint32_t vm = ((rows >> row) & 1) ? ~0u : 0u;
#pragma unroll
        for (int c = 0; c < kALoads; ++c) raw[c] = make_uint4(raw[c].x & vm, raw[c].y & vm, raw[c].z & vm, raw[c].w & vm);
        float2 vf[kAPairs];
#pragma unroll
        for (int c = 0; c < kALoads; ++c) unpack16x2<T>(raw[c], vf + c * (kAPairs / kALoads));
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          const float wv = __shfl_sync(kFull, w, (lane & 16) | ((tt * G + hh) << kAPlain));
          const float2 w2 = make_float2(wv, wv);
#pragma unroll
          for (int i = 0; i < kAPairs; ++i) A.o[hh][i] = __ffma2_rn(w2, vf[i], A.o[hh][i]);
        }
      }
    }
  }

  // The warp's state -> one partial summary per head at dst ([G][kPartStride]):
  // the two half-warps brought to a common maximum and summed.  only >= 0:
  // that head's partial alone, at dst.
  __device__ static void att_finish(Att &A, float *dst, int only = -1) {
    const int lane = lane_id(), sub = lane & 15, hw = lane >> 4;
    const int idx = sub >> kAPlain, hm = idx % G;
    const float l_grp = head_sum(A.l_mine);  // this half-warp's sum for head hm
    float M[G];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      M[hh] = fmaxf(A.mrun[hh], __shfl_xor_sync(kFull, A.mrun[hh], 16));
      const float f = ex2(A.mrun[hh] - M[hh]);
#pragma unroll
      for (int i = 0; i < kAPairs; ++i) {
        float2 x = __fmul2_rn(A.o[hh][i], make_float2(f, f));
        x.x += __shfl_xor_sync(kFull, x.x, 16);
        x.y += __shfl_xor_sync(kFull, x.y, 16);
        A.o[hh][i] = x;
      }
    }
    float Mm = M[0];
#pragma unroll
    for (int hh = 1; hh < G; ++hh) Mm = hm == hh ? M[hh] : Mm;
    float L = l_grp * ex2(A.m_mine - Mm);
    L += __shfl_xor_sync(kFull, L, 16);
    if (hw == 0) {
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        if (only >= 0 && hh != only) continue;
        float *o = dst + (only >= 0 ? 0 : hh * kPartStride) + sub * 8;
        *reinterpret_cast<float4 *>(o) = make_float4(A.o[hh][0].x, A.o[hh][0].y, A.o[hh][1].x, A.o[hh][1].y);
        *reinterpret_cast<float4 *>(o + 4) = make_float4(A.o[hh][2].x, A.o[hh][2].y, A.o[hh][3].x, A.o[hh][3].y);
      }
      if ((sub & ((1 << kAPlain) - 1)) == 0 && idx < G && (only < 0 || hm == only))  // one lane per head
        *reinterpret_cast<float2 *>(dst + (only >= 0 ? 0 : hm * kPartStride) + kHeadDim) = make_float2(Mm, L);
    }
  }

  // R(pos) q~ * log2(e)/sqrt(d) of the G heads of unit u, the lane's dims
  // [8 sub, 8 sub + 8) (explicit roundings keep the result identical
  // wherever it is computed).
  // R(pos) q~ * log2(e)/sqrt(d) of the G heads of unit u, the lane's dims
  // [8 sub, 8 sub + 8), from the query rows in global memory or (qe) in a
  // warp's query entry holding the G rows back to back.  Every pair (a, b)
  // of a 2x2 rotation becomes a' = a cos - b sin, b' = b cos + a sin; a lane
  // computes its own dims x from its partner dims y with signed sines (the
  // explicit roundings keep the result identical wherever it is computed).
  __device__ static void load_query(const StepParams &p, const Smem &S, int u, float2 (&q)[G][kAPairs],
                                    const uint8_t *qe = nullptr) {
    const int lane = lane_id(), sub = lane & 15;
    const int b = u / p.Hkv, g = u - b * p.Hkv;
    const bool half = p.rope_mode == MAC_ROPE_HALF, none = p.rope_mode == MAC_ROPE_NONE;
    const int d0 = sub * 8, dp = (d0 + kHeadDim / 2) & (kHeadDim - 1);  // own dims, partner dims (half mode)
    float c[8], sn[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      // half: pair (j, j + d/2), own dims below d/2 are a; interleaved: pair (2j, 2j + 1)
      const int j = half ? (d0 + i) & (kHeadDim / 2 - 1) : (d0 + i) >> 1;
      float2 cs = make_float2(1.f, 0.f);
      if (!none) {
        if (S.rope) cs = S.rope[b * (kHeadDim / 2) + j];
        else rope_angle(qpos(p, b), p.rope_f[j], &cs.x, &cs.y);
      }
      const bool is_a = half ? d0 < kHeadDim / 2 : (i & 1) == 0;
      c[i] = cs.x;
      sn[i] = is_a ? -cs.y : cs.y;
    }
    bool bad = false;
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      const int64_t e0 = ((int64_t)b * p.Hq + g * G + hh) * p.q_stride + p.q_offset;
      const T *row = qe ? reinterpret_cast<const T *>(qe + hh * kRow) : reinterpret_cast<const T *>(p.q) + e0;
      float x[8], y[8];
#pragma unroll
      for (int k = 0; k < kALoads; ++k) {
        float2 f[kAPairs / kALoads], h[kAPairs / kALoads];
        const uint4 *o4 = reinterpret_cast<const uint4 *>(row + d0) + k;
        const uint4 *p4 = reinterpret_cast<const uint4 *>(row + dp) + k;
        unpack16x2<T>(qe ? *o4 : __ldg(o4), f);
        unpack16x2<T>(half ? (qe ? *p4 : __ldg(p4)) : make_uint4(0, 0, 0, 0), h);
#pragma unroll
        for (int i = 0; i < kAPairs / kALoads; ++i) {
          x[k * 8 / kALoads + 2 * i] = f[i].x;
          x[k * 8 / kALoads + 2 * i + 1] = f[i].y;
          y[k * 8 / kALoads + 2 * i] = h[i].x;
          y[k * 8 / kALoads + 2 * i + 1] = h[i].y;
        }
      }
      float r[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        bad |= !isfinite(x[i]);
        const float yy = half ? y[i] : none ? 0.f : x[i ^ 1];
        r[i] = none ? __fmul_rn(x[i], p.q_scale)
                    : __fmul_rn(__fadd_rn(__fmul_rn(x[i], c[i]), __fmul_rn(yy, sn[i])), p.q_scale);
      }
#pragma unroll
      for (int i = 0; i < kAPairs; ++i) q[hh][i] = make_float2(r[2 * i], r[2 * i + 1]);
    }
    if (bad) set_status(p.ctl, MAC_DEV_NONFINITE_Q);
  }

  // ---------------------------------------------------------------------
  // match
  // ---------------------------------------------------------------------
  // The squared distance over the lane's 8 dims of one half of a row (exact
  // bf16 differences, squares summed in a pairwise tree).
  __device__ static float half_dist(const float2 (&qv)[4], const uint8_t *src) {
    float2 df[4];
    if constexpr (sizeof(T) == 2) {
      // b - q straight from the bf16 element (one mixed-precision
      // subtraction each): the negation of the difference, same square
      const uint4 raw = *reinterpret_cast<const uint4 *>(src);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int k = 0; k < 4; ++k)
        df[k] = make_float2(bf16_minus_f32((uint16_t)(w[k] & 0xffffu), qv[k].x),
                            bf16_minus_f32((uint16_t)(w[k] >> 16), qv[k].y));
    } else {
      float2 e[4];
#pragma unroll
      for (int c = 0; c < kHalfLoads; ++c)
        unpack16x2<T>(*reinterpret_cast<const uint4 *>(src + c * 16), e + c * (4 / kHalfLoads));
#pragma unroll
      for (int k = 0; k < 4; ++k) df[k] = __fadd2_rn(qv[k], make_float2(-e[k].x, -e[k].y));
    }
    const float2 t0 = __ffma2_rn(df[2], df[2], __fmul2_rn(df[0], df[0]));
    const float2 t1 = __ffma2_rn(df[3], df[3], __fmul2_rn(df[1], df[1]));
    const float2 t = __fadd2_rn(t0, t1);
    return __fadd_rn(t.x, t.y);
  }
  // v[k]: this lane's part of row k of its group -> the lane's row total
  // (row sub >> (3 - kLogMRG)): reduce-scatter over the 8 lanes, then plain
  // butterflies (a pairwise tree of the 8 lanes' parts).
  __device__ static float group_reduce(float (&v)[kMRG]) {
#pragma unroll
    for (int lev = 0; lev < kLogMRG; ++lev) {
      const int off = 4 >> lev;
      const bool up = (threadIdx.x & off) != 0;
      const int half = kMRG >> (lev + 1);
#pragma unroll
      for (int i = 0; i < kMRG / 2; ++i) {
        if (i < half) {
          const float send = up ? v[i] : v[i + half];
          const float keep = up ? v[i + half] : v[i];
          v[i] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, off));
        }
      }
    }
    float D = v[0];
#pragma unroll
    for (int lev = kLogMRG; lev < 3; ++lev) D = __fadd_rn(D, __shfl_xor_sync(kFull, D, 4 >> lev));
    return D;
  }
  // the stage row whose distance this lane finishes
  __device__ static int match_row(int lane) { return (lane >> 3) + 4 * (((lane & 7) >> (3 - kLogMRG)) & (kMRG - 1)); }
  // One stage of ring rows (cnt of them): the lane's candidate (distance,
  // position pk) joins its running best.
  __device__ static void match_stage(const uint8_t *buf, int cnt, const float2 (&qlo)[4], const float2 (&qhi)[4],
                                     int pk, int pos_lo, int pos_hi, float &bd, int &bp) {
    const int lane = lane_id(), grp = lane >> 3, sub = lane & 7;
    float lo[kMRG], hi[kMRG];
#pragma unroll
    for (int k = 0; k < kMRG; ++k) {
      const int r = grp + 4 * k;
      const uint8_t *row = buf + (size_t)(r < cnt ? r : cnt - 1) * kRow;
      lo[k] = half_dist(qlo, row + sub * 8 * kES);
      hi[k] = half_dist(qhi, row + kRow / 2 + sub * 8 * kES);
    }
    const float D = __fadd_rn(group_reduce(lo), group_reduce(hi));
    if (match_row(lane) < cnt && pk >= pos_lo && pk <= pos_hi && better(D, pk, bd, bp)) {
      bd = D;
      bp = pk;
    }
  }

  // ---------------------------------------------------------------------
  // phase A: window tiles and match items, round-robin over all warps
  // ---------------------------------------------------------------------
  __device__ static int n_units(const StepParams &p) { return p.B * p.Hkv; }
  __device__ static int match_cph(const StepParams &p) { return (p.K + kIR - 1) / kIR; }
  __device__ static int64_t n_window_items(const StepParams &p) { return (int64_t)n_units(p) * p.tc.nt; }
  __device__ static int64_t n_items(const StepParams &p) {
    return n_window_items(p) + (p.mode == MODE_DECODE ? (int64_t)p.B * p.Hq * match_cph(p) : 0);
  }
  // One streamed item: a window tile (kind 1: unit u, tokens [lo, hi], all
  // heads), a match item (kind 2: head u, ring rows [lo, hi)), or a boundary
  // piece (kind 3: unit u, tokens [lo, hi] for head hm alone, into the
  // warp's slot of S.bd); kind -1: none.
  struct Item {
    int64_t i;
    int kind, u, lo, hi, hm;
  };
  __device__ static Item no_item() {
    Item it;
    it.i = 0;
    it.kind = -1;
    it.u = it.lo = it.hm = 0;
    it.hi = -1;
    return it;
  }
  // phase-A item i: the window tiles of every unit, then the match items
  __device__ static Item item_a(const StepParams &p, const Smem &S, int64_t i) {
    Item it = no_item();
    it.i = i;
    const int64_t nw = n_window_items(p);
    if (i < 0 || i >= n_items(p)) return it;
    if (i < nw) {
      const int u = (int)((uint32_t)i / (uint32_t)p.tc.nt), t = (int)i - u * p.tc.nt;
      it.kind = 1;
      it.u = u;
      tile_range(p, S.um[u], t, &it.lo, &it.hi);
    } else {
      const int cph = match_cph(p);
      const int mi = (int)(i - nw), bh = (int)((uint32_t)mi / (uint32_t)cph);
      it.kind = 2;
      it.u = bh;
      it.lo = (mi - bh * cph) * kIR;
      it.hi = min(p.K, it.lo + kIR);
    }
    return it;
  }
  // The boundary piece of owned head k (none when the head misses or its
  // band starts on a tile boundary): the band [lo, m - r] of a hit at p
  // starts at lo = p - r + 1 inside band tile j; the piece is [lo, end of
  // tile j] for that head alone.  *nbt: the band tiles the head takes whole.
  __device__ static Item boundary_item(const StepParams &p, const Smem &S, int bh, int pos, int *nbt) {
    Item it = no_item();
    const int b = bh / p.Hq, h = bh - b * p.Hq, g = h / G, u = b * p.Hkv + g;
    const int m = S.um[u];
    *nbt = p.tc.nbw;
    if (pos < 1 || m <= 0) return it;
    const int lo = max(lb(p), pos - p.r + 1);
    if (lo > m - p.r) {
      *nbt = 0;
      return it;
    }
    const int j = (m - p.r - lo) / kTT;
    int tlo, thi;
    tile_range(p, m, j, &tlo, &thi);
    *nbt = lo == tlo ? j + 1 : j;
    if (lo == tlo) return it;
    it.kind = 3;
    it.u = u;
    it.lo = lo;
    it.hi = thi;
    it.hm = h - g * G;
    return it;
  }
  // stage s of an item
  __device__ static Desc stage_desc(const StepParams &p, const Item &it, int s) {
    Desc d;
    d.kind = it.kind == 2 ? 2 : 1;
    d.u = it.u;
    if (it.kind != 2) {
      d.a = it.lo + s * kStTok;
      d.cnt = min(it.hi - d.a + 1, kStTok);
      d.keep = it.kind == 1;
    } else {
      d.a = it.lo + s * kStRows;
      d.cnt = min(it.hi - d.a, kStRows);
      if (d.cnt <= 0) d.kind = 0;
      d.pc = d.kind == 2 && (p.K & 3) == 0 && (d.cnt & 3) == 0;
    }
    return d;
  }
  // the query an item needs: its unit (window, boundary) or head (match)
  __device__ static int query_key(const Item &it) { return it.kind == 2 ? -1 - it.u : it.u; }

  // The streaming loop of one round, one copy of the per-stage code for all
  // rounds: round 0 streams this warp's contiguous share of the phase-A
  // items; round r >= 1 the boundary piece of owned head (r-1) kWarps + w.
  // One iteration per stage; the copies run up to kStages stages ahead.
  // Consecutive items of a warp mostly share their query; an item whose
  // query differs from the one before brings it along with its first stage
  // (into the warp's next query entry), so the loop waits on nothing but its
  // stages.  Without query entries (no room in shared memory) the query is
  // read from global memory.
  __device__ static void stream(const StepParams &p, const Smem &S, Ring &R, int rnd, int h0, int hstep, int nown) {
    const int lane = lane_id(), w = warp_id(), P = gridDim.x, NW = P * kWarps;
    const int gw = w * P + blockIdx.x;
    int64_t i_beg = 0, i_end = 0;
    if (rnd == 0) {
      const int64_t na = n_items(p);
      i_beg = (int64_t)(((unsigned long long)gw * (unsigned long long)na) / (unsigned)NW);
      i_end = (int64_t)(((unsigned long long)(gw + 1) * (unsigned long long)na) / (unsigned)NW);
    } else {
      const int k = (rnd - 1) * kWarps + w;
      i_end = k < nown ? 1 : 0;
    }
    auto get = [&](int64_t i) -> Item {
      if (i >= i_end) return no_item();
      if (rnd == 0) return item_a(p, S, i);
      const int k = (rnd - 1) * kWarps + w, bh = h0 + k * hstep;
      int nbt;
      Item it = boundary_item(p, S, bh, k < kOwnMax ? S.dec[k] : decision(p, S, bh), &nbt);
      it.i = i;
      return it;
    };
    int32_t id[2];
    // fetch side: the next stage to copy; it attaches the query of each
    // item whose query differs from the last
    Item fi = get(i_beg);
    int fs = 0, f_key = 0x7fffffff, f_e = 1;
    Desc nx;
    bool have_nx = false;
    auto fetch_next = [&]() {
      have_nx = fi.kind >= 0;
      if (!have_nx) return;
      nx = stage_desc(p, fi, fs);
      if (fs == 0 && query_key(fi) != f_key) {
        f_key = query_key(fi);
        f_e ^= 1;
        nx.qe = f_e;
      }
      if (++fs == kItemStages) {
        fs = 0;
        fi = get(fi.i + 1);
      }
      load_ids(p, nx, id);
    };
    fetch_next();
    Att A;
    float2 q[G][kAPairs];
    float2 qlo[4], qhi[4];
    float bd = INFINITY;
    int bp = -1, pos_lo = 1, pos_hi = 0;
    int c_key = 0x7fffffff, c_e = 1;  // the query in registers, its entry
    Item ci = get(i_beg);
    int cs = 0;  // the stage of ci to consume
#pragma unroll 1
    for (;;) {
      // keep kStages copies in flight
#pragma unroll 1
      while (have_nx && R.issued - R.used < (uint32_t)kStages) {
        issue(p, R, nx, id);
        fetch_next();
      }
      if (ci.kind < 0 || *S.abort) break;
      if (cs == 0) {
        if (ci.kind == 2) {
          const int m = S.um[(ci.u / p.Hq) * p.Hkv];
          pos_lo = m > 0 ? max(1, m - p.K) : 1;
          pos_hi = m > 0 ? m - 1 : 0;
          bd = INFINITY;
          bp = -1;
        } else {
          att_init(A);
        }
      }
      const Desc d = stage_desc(p, ci, cs);
      const int r = match_row(lane);
      int pk = 0;
      if (d.kind == 2 && !d.pc)  // the position of the row this lane finishes, read directly
        pk = __ldg(p.ring_pos + (int64_t)(d.u / p.Hq) * p.K + d.a + (r < d.cnt ? r : d.cnt - 1));
      const uint32_t n = R.used;
      const bool ok = wait_stage(p, S, R, n);
      const int key = query_key(ci);
      if (cs == 0 && key != c_key) {
        // the item's query came with its first stage (or is read directly)
        c_e ^= 1;
        c_key = key;
        const uint8_t *qe = R.qbuf ? R.qbuf + (size_t)c_e * kQE : nullptr;
        if (ci.kind != 2) {
          load_query(p, S, ci.u, q, qe);
        } else {
          const T *row = qe ? reinterpret_cast<const T *>(qe)
                            : reinterpret_cast<const T *>(p.q) + (int64_t)ci.u * p.q_stride + p.q_offset;
#pragma unroll
          for (int c = 0; c < kHalfLoads; ++c) {
            const uint4 *lo4 = reinterpret_cast<const uint4 *>(row + (lane & 7) * 8) + c;
            const uint4 *hi4 = reinterpret_cast<const uint4 *>(row + kHeadDim / 2 + (lane & 7) * 8) + c;
            unpack16x2<T>(qe ? *lo4 : __ldg(lo4), qlo + c * (4 / kHalfLoads));
            unpack16x2<T>(qe ? *hi4 : __ldg(hi4), qhi + c * (4 / kHalfLoads));
          }
        }
      }
      if (ok) {
        const uint8_t *buf = stage_buf(R, n);
        if (d.kind == 1 && d.cnt > 0) {
          // a boundary piece counts for its head alone
          const int hm = ((lane & 15) >> kAPlain) % G;
          const bool mine = ci.kind != 3 || hm == ci.hm;
          att_stage(A, q, buf, d.a, R.rows[n % kStages], mine ? d.a : 1, mine ? d.a + d.cnt - 1 : 0);
        } else if (d.kind == 2) {
          if (d.pc)
            pk = reinterpret_cast<const int32_t *>(R.pside + (size_t)(n % kStages) * kPosBytes)[r < d.cnt ? r : d.cnt - 1];
          match_stage(buf, d.cnt, qlo, qhi, pk, pos_lo, pos_hi, bd, bp);
        }
      }
      R.used++;
      done_with_stage();
      if (++cs < kItemStages) continue;
      // the item is done
      cs = 0;
      if (ci.kind == 1) {
        const int u = ci.u, t = (int)(ci.i - (int64_t)u * p.tc.nt);
        att_finish(A, p.part_w + ((size_t)u * p.tc.nt + t) * G * kPartStride);
      } else if (ci.kind == 3) {
        att_finish(A, S.bd + (size_t)w * kPartStride, ci.hm);
      } else {
        // the warp's best joins the head's minimum
#pragma unroll
        for (int off = 1; off <= 16; off <<= 1) {
          const float d2 = __shfl_xor_sync(kFull, bd, off);
          const int p2 = __shfl_xor_sync(kFull, bp, off);
          if (better(d2, p2, bd, bp)) {
            bd = d2;
            bp = p2;
          }
        }
        if (lane == 0 && bp >= 1) atomicMax(&S.best[ci.u], pack_best(bd, bp));
      }
      ci = get(ci.i + 1);
    }
  }

  // ---------------------------------------------------------------------
  // decisions and the long-band layout
  // ---------------------------------------------------------------------
  // The decision of head bh: the matched position, or -1 (miss).
  __device__ static int decision(const StepParams &p, const Smem &S, int bh) {
    if (p.mode != MODE_DECODE) return -1;
    const int m = S.um[(bh / p.Hq) * p.Hkv];
    const unsigned long long inv = __ldcg(&S.best[bh]);
    if (inv == 0ull || m <= 0 || m < p.min_context) return -1;
    const unsigned long long key = ~inv;
    const float d = __uint_as_float((uint32_t)(key >> 32));
    return d < p.thr2 ? (int)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull)) : -1;
  }
  // Long-band length of unit u: tokens [lb, win_start - 1] of a unit with a
  // missing head.
  __device__ static int64_t long_len(const StepParams &p, const Smem &S, int u, bool miss) {
    const int m = S.um[u];
    if (m <= 0 || !miss) return 0;
    return max(0, win_start(p, m) - lb(p));
  }

  // Exclusive scan of one value per thread, in thread order, and the total.
  // All threads call it; it holds two barriers.
  __device__ static long long block_scan(const Smem &S, long long x, long long *total) {
    const int lane = lane_id(), warp = warp_id();
    long long xi = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(kFull, xi, o);
      if (lane >= o) xi += y;
    }
    if (lane == 31) S.scan[warp] = xi;
    block_sync();
    long long base = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const long long v = S.scan[w];
      base += w < warp ? v : 0;
      tot += v;
    }
    block_sync();
    *total = tot;
    return base + xi - x;
  }

  // Heads owned (merged) by this CTA, out of N: bh with floor(bh P / N) == c
  // (N <= P), or bh = c, c + P, ... (N > P); own_index: the head's rank among
  // them, -1 when not owned here or beyond the kOwnMax whose decisions are
  // kept.
  static constexpr int kOwnMax = 16;
  __device__ static void own_range(int U, int *u0, int *u_end, int *step) {
    const int P = gridDim.x, c = blockIdx.x;
    *u0 = U <= P ? (c * U + P - 1) / P : c;
    *u_end = U <= P ? ((c + 1) * U + P - 1) / P : U;
    *step = U <= P ? 1 : P;
  }
  __device__ static int own_index(int U, int u) {
    int u0, u_end, step;
    own_range(U, &u0, &u_end, &step);
    if (u < u0 || u >= u_end || (u - u0) % step != 0) return -1;
    const int k = (u - u0) / step;
    return k < kOwnMax ? k : -1;
  }

  // Every unit's long-band offset (units end to end) and the number of CTAs
  // they are cut over; the same in every CTA.  Ends with a barrier.
  __device__ static void layout_long(const StepParams &p, const Smem &S) {
    const int U = n_units(p);
    long long carry = 0;
#pragma unroll 1
    for (int base = 0; base < U; base += kThreads) {
      const int u = base + threadIdx.x;
      long long x = 0;
      if (u < U) {
        bool miss = p.mode != MODE_DECODE;
        const int b = u / p.Hkv, g = u - b * p.Hkv;
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          const int bh = b * p.Hq + g * G + hh, pos = decision(p, S, bh);
          const int k = own_index(p.B * p.Hq, bh);
          miss |= pos < 1;
          if (k >= 0) S.dec[k] = pos;
        }
        x = long_len(p, S, u, miss);
      }
      long long tot;
      const long long ex = block_scan(S, x, &tot);
      if (u < U) S.off[u + 1] = carry + ex + x;
      carry += tot;
    }
    if (threadIdx.x == 0) {
      S.off[0] = 0;
      *S.ntok = carry;
      const long long want = (carry + kMinSpan - 1) / kMinSpan;
      *S.Pl = carry > 0 ? (int)(want < (long long)gridDim.x ? want : (long long)gridDim.x) : 0;
    }
    block_sync();
  }
  // span of CTA c on the long-band axis: [span(c), span(c + 1)) (c < Pl)
  __device__ static int64_t span(const Smem &S, int c) {
    const int64_t tot = *S.ntok;
    const int Pl = *S.Pl;
    return c >= Pl ? tot : (int64_t)(((unsigned long long)c * (unsigned long long)tot) / (unsigned long long)Pl);
  }
  // the CTA whose span holds long-band index x (0 <= x < T): the largest c
  // with span(c) <= x
  __device__ static int cta_of(const Smem &S, int64_t x) {
    return (int)((((unsigned long long)x + 1) * (unsigned long long)*S.Pl - 1) / (unsigned long long)*S.ntok);
  }
  // the last unit u with off[u] <= x
  __device__ static int unit_of(const StepParams &p, const Smem &S, int64_t x) {
    const int U = n_units(p);
    int lo = 0;
#pragma unroll 1
    for (int s = U > 1 ? 1 << (31 - __clz(U - 1)) : 0; s >= 1; s >>= 1) {
      const int t = lo + s;
      if (t < U && S.off[t] <= x) lo = t;
    }
    return lo;
  }
  // unit u's CTA run [*c0, *c1] (empty: *c1 < *c0)
  __device__ static void long_run(const Smem &S, int u, int *c0, int *c1) {
    const int64_t a = S.off[u], z = S.off[u + 1];
    if (z <= a) {
      *c0 = 0;
      *c1 = -1;
      return;
    }
    *c0 = cta_of(S, a);
    *c1 = cta_of(S, z - 1);
  }
  // long-band entries of unit u's merge: CTA pieces, or CTA groups
  __device__ static bool grouped(int c0, int c1) { return c1 - c0 + 1 > kGroupCtas; }
  __device__ static int long_entries(int c0, int c1) {
    if (c1 < c0) return 0;
    return grouped(c0, c1) ? c1 / kGroupCtas - c0 / kGroupCtas + 1 : c1 - c0 + 1;
  }
  __device__ static const float *long_entry(const StepParams &p, int u, int c0, int c1, int i, int hh) {
    if (grouped(c0, c1)) return p.part_g + ((size_t)(u + c0 / kGroupCtas + i) * G + hh) * kPartStride;
    return p.part_c + ((size_t)(u + c0 + i) * G + hh) * kPartStride;
  }

  // ---------------------------------------------------------------------
  // merges
  // ---------------------------------------------------------------------
  template <int N>
  __device__ static void load_dims(const float *src, float (&v)[N]) {
    if constexpr (N == 4) {
      const float4 x = __ldcg(reinterpret_cast<const float4 *>(src));
      v[0] = x.x;
      v[1] = x.y;
      v[2] = x.z;
      v[3] = x.w;
    } else if constexpr (N == 2) {
      const float2 x = __ldcg(reinterpret_cast<const float2 *>(src));
      v[0] = x.x;
      v[1] = x.y;
    } else {
      v[0] = __ldcg(src);
    }
  }
  template <int N>
  __device__ static void store_dims(float *dst, const float (&v)[N]) {
    if constexpr (N == 4)
      *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
    else if constexpr (N == 2)
      *reinterpret_cast<float2 *>(dst) = make_float2(v[0], v[1]);
    else
      dst[0] = v[0];
  }
  // the weight of a member (m, l) in a state at maximum M
  // (a member with nothing in it, l == 0 or m == -inf, weighs 0)
  __device__ static float mweight(float m, float l, float M) { return l > 0.f && m > -INFINITY ? ex2(m - M) : 0.f; }

  // A log-domain state (base 2) over this lane's dims: maximum, sum, weighted values.
  struct Cls {
    float M, L, O[kDL];
  };
  // The states of one head's list for this lane's dims [dl, dl + kDL):
  // entries 0..n-1 (entry(i) -> partial, or null: empty), the first nb of
  // the band class, the rest of the tail class.  Each class is summed at its
  // maximum over the entries holding tokens.  Lane j holds entry j's
  // pointer, maximum and sum; up to kBatch entries' outputs are in flight at
  // once, so a list of up to kBatch entries costs one trip to L2.
  template <class F>
  __device__ static void merge_list(int n, int nb, F entry, int dl, Cls &band, Cls &tail) {
    constexpr int kBatch = 8;
    const int lane = lane_id();
    band.M = tail.M = -INFINITY;
    band.L = tail.L = 0.f;
#pragma unroll
    for (int i = 0; i < kDL; ++i) band.O[i] = tail.O[i] = 0.f;
#pragma unroll 1
    for (int base = 0; base < n; base += 32) {
      const int cnt = min(32, n - base);
      const float *src = lane < cnt ? entry(base + lane) : nullptr;
      if (!src) src = g_zero_partial;
      const float2 ml = __ldcg(reinterpret_cast<const float2 *>(src + kHeadDim));
      const unsigned long long sp = reinterpret_cast<unsigned long long>(src);
      float ov[kBatch][kDL];
#pragma unroll
      for (int k = 0; k < kBatch; ++k)
        load_dims<kDL>(reinterpret_cast<const float *>(__shfl_sync(kFull, sp, k)) + dl, ov[k]);
      const bool isb = base + lane < nb;
      float mb = isb && ml.y > 0.f ? ml.x : -INFINITY, mt = !isb && ml.y > 0.f ? ml.x : -INFINITY;
#pragma unroll
      for (int o2 = 16; o2 >= 1; o2 >>= 1) {
        mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, o2));
        mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, o2));
      }
      // what earlier rounds summed, at the new maxima
      mb = fmaxf(band.M, mb);
      mt = fmaxf(tail.M, mt);
      const float rb = mweight(band.M, band.L, mb), rt = mweight(tail.M, tail.L, mt);
      band.L *= rb;
      tail.L *= rt;
#pragma unroll
      for (int i = 0; i < kDL; ++i) {
        band.O[i] *= rb;
        tail.O[i] *= rt;
      }
      band.M = mb;
      tail.M = mt;
      const float wgt = mweight(ml.x, ml.y, isb ? band.M : tail.M);
      const float wb = isb ? wgt : 0.f, wt = isb ? 0.f : wgt;
      float lbs = wb * ml.y, lts = wt * ml.y;
#pragma unroll
      for (int o2 = 16; o2 >= 1; o2 >>= 1) {
        lbs += __shfl_xor_sync(kFull, lbs, o2);
        lts += __shfl_xor_sync(kFull, lts, o2);
      }
      band.L += lbs;
      tail.L += lts;
#pragma unroll 1
      for (int k0 = 0; k0 < cnt; k0 += kBatch) {
        if (k0 > 0) {
#pragma unroll
          for (int k = 0; k < kBatch; ++k)
            load_dims<kDL>(reinterpret_cast<const float *>(__shfl_sync(kFull, sp, (k0 + k) & 31)) + dl, ov[k]);
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          // past the round's entries the batch wraps onto lanes already summed
          const int j = (k0 + k) & 31;
          const bool in = k0 + k < cnt;
          float xb = __shfl_sync(kFull, wb, j), xt = __shfl_sync(kFull, wt, j);
          xb = in ? xb : 0.f;
          xt = in ? xt : 0.f;
#pragma unroll
          for (int i = 0; i < kDL; ++i) {
            band.O[i] = fmaf(xb, ov[k][i], band.O[i]);
            tail.O[i] = fmaf(xt, ov[k][i], tail.O[i]);
          }
        }
      }
    }
  }
  // a (+)= x, each state at its own maximum
  __device__ static void join(Cls &a, float xm, float xl, const float (&xo)[kDL]) {
    const float M = fmaxf(a.L > 0.f ? a.M : -INFINITY, xl > 0.f ? xm : -INFINITY);
    const float wa = mweight(a.M, a.L, M), wx = mweight(xm, xl, M);
    a.L = wa * a.L + wx * xl;
#pragma unroll
    for (int i = 0; i < kDL; ++i) a.O[i] = wa * a.O[i] + wx * xo[i];
    a.M = M;
  }

  // The owner's merge of one head bh by all the CTA's warps: before the long
  // bands (pass 0) a hit or a miss of a unit without a long band, after them
  // (pass 1) a miss of a unit with one.  AS = [cached] (+) [boundary] (+)
  // band tiles [0, nbt) (+) long-band entries; the output AS (+) tail tiles
  // (+) sink tiles; the rectified summary AS_{1:m-r} goes to the ring slot
  // of position m (fused append) or to the staging area.  Warp w sums list
  // entries w, w + 8, ... (4 dims per lane) per class; the CTA then combines
  // the warps' states in a fixed order.  A hit whose band starts inside a
  // window tile has a boundary piece, streamed before the merge into warp
  // bd_w's slot of S.bd.  pos: the head's decision (-2: not known yet).
  // All threads call it.
  struct St {
    float M, L, O[4];
  };
  __device__ static void st_join(St &a, float xm, float xl, const float4 &xo) {
    const float M = fmaxf(a.L > 0.f ? a.M : -INFINITY, xl > 0.f ? xm : -INFINITY);
    const float wa = mweight(a.M, a.L, M), wx = mweight(xm, xl, M);
    a.L = wa * a.L + wx * xl;
    a.O[0] = wa * a.O[0] + wx * xo.x;
    a.O[1] = wa * a.O[1] + wx * xo.y;
    a.O[2] = wa * a.O[2] + wx * xo.z;
    a.O[3] = wa * a.O[3] + wx * xo.w;
    a.M = M;
  }
  __device__ static void merge_one(const StepParams &p, const Smem &S, int bh, bool long_pass, int pos, int bd_w) {
    const int b = bh / p.Hq, h = bh - b * p.Hq, g = h / G, hh = h - g * G, u = b * p.Hkv + g;
    const int lane = lane_id(), w = warp_id(), tid = threadIdx.x;
    const bool decode = p.mode == MODE_DECODE;
    if (pos == -2) pos = decision(p, S, bh);
    int c0, c1;
    long_run(S, u, &c0, &c1);
    const bool late = pos < 1 && c1 >= c0;
    if (late != long_pass) return;
    const int m = S.um[u];
    if (m <= 0) {
      // a length outside the cache: zero output, no append
      if (tid < kHeadDim) p.out[(int64_t)bh * kHeadDim + tid] = 0.f;
      if (tid == 0) {
        if (p.out_lse) p.out_lse[bh] = -INFINITY;
        if (p.match_pos_out) p.match_pos_out[bh] = -1;
      }
      block_sync();
      return;
    }
    int nbt;
    const bool has_bd = boundary_item(p, S, bh, pos, &nbt).kind == 3 && !long_pass;
    if (pos >= 1) {
      c0 = 0;
      c1 = -1;
    } else {
      nbt = p.tc.nbw;
    }
    unsigned long long *tr = p.trace && lane == 0 && w <= 1 ? p.trace + (size_t)blockIdx.x * kTracePoints : nullptr;
    if (tr && w == 0) tr[18] = globaltimer();
    // the cached rectified summary of a hit (a state of sum 1 at its ln-LSE), by warp 1
    const int64_t cslot = (int64_t)bh * p.K + (pos >= 1 ? pos % p.K : 0);
    float c_lse = 0.f;
    float4 c_o = make_float4(0.f, 0.f, 0.f, 0.f);
    if (pos >= 1 && w == 1) {
      c_lse = __ldcg(p.ring_lse + cslot);
      c_o = __ldcg(reinterpret_cast<const float4 *>(p.ring_o + cslot * kHeadDim) + lane);
    }
    const int nl = long_entries(c0, c1);
    const int nt = p.tc.ntt + (p.sink_piece ? p.tc.nsk : 0);
    const int n = nbt + nl + nt, nb = nbt + nl;
    const float *tiles = p.part_w + (size_t)u * p.tc.nt * G * kPartStride + hh * kPartStride;
    auto entry = [&](int i) -> const float * {
      if (i < nbt) return tiles + (size_t)i * G * kPartStride;
      i -= nbt;
      if (i < nl) return long_entry(p, u, c0, c1, i, hh);
      i -= nl;
      return tiles + (size_t)(p.tc.nbw + i) * G * kPartStride;
    };
    St band, tail;
    band.M = tail.M = -INFINITY;
    band.L = tail.L = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) band.O[i] = tail.O[i] = 0.f;
    constexpr int kE = 8;  // entries a warp has in flight
#pragma unroll 1
    for (int i0 = w; i0 < n; i0 += kWarps * kE) {
      float2 ml[kE];
      float4 ov[kE];
#pragma unroll
      for (int e = 0; e < kE; ++e) {
        const int i = i0 + e * kWarps;
        const float *src = i < n ? entry(i) : g_zero_partial;
        ml[e] = __ldcg(reinterpret_cast<const float2 *>(src + kHeadDim));
        ov[e] = __ldcg(reinterpret_cast<const float4 *>(src) + lane);
      }
#pragma unroll
      for (int e = 0; e < kE; ++e) {
        const int i = i0 + e * kWarps;
        if (i < nb) st_join(band, ml[e].x, ml[e].y, ov[e]);
        else if (i < n) st_join(tail, ml[e].x, ml[e].y, ov[e]);
      }
    }
    if (pos >= 1 && w == 1) st_join(band, c_lse * kLog2e, 1.f, c_o);
    if (tr) tr[w == 0 ? 13 : 19] = globaltimer();
    if (has_bd && w == 0) {
      const float *x = S.bd + (size_t)bd_w * kPartStride;
      st_join(band, x[kHeadDim], x[kHeadDim + 1], reinterpret_cast<const float4 *>(x)[lane]);
    }
    // the warps' states, in warp 7's idle stage ring
    float *red = reinterpret_cast<float *>(S.stage + (size_t)7 * kStages * kStageBytes);
#pragma unroll
    for (int cls = 0; cls < 2; ++cls) {
      const St &st = cls ? tail : band;
      float *d = red + (w * 2 + cls) * kPartStride;
      reinterpret_cast<float4 *>(d)[lane] = make_float4(st.O[0], st.O[1], st.O[2], st.O[3]);
      if (lane == 0) *reinterpret_cast<float2 *>(d + kHeadDim) = make_float2(st.M, st.L);
    }
    if (tr && w == 0) tr[14] = globaltimer();
    block_sync();
    if (tr && w == 0) tr[15] = globaltimer();
    if (tid < kHeadDim) {
      float MB = -INFINITY, MT = -INFINITY;
#pragma unroll
      for (int ww = 0; ww < kWarps; ++ww) {
        const float *bs = red + (ww * 2) * kPartStride, *ts = bs + kPartStride;
        if (bs[kHeadDim + 1] > 0.f) MB = fmaxf(MB, bs[kHeadDim]);
        if (ts[kHeadDim + 1] > 0.f) MT = fmaxf(MT, ts[kHeadDim]);
      }
      float LB = 0.f, OB = 0.f, LT = 0.f, OT = 0.f;
#pragma unroll
      for (int ww = 0; ww < kWarps; ++ww) {
        const float *bs = red + (ww * 2) * kPartStride, *ts = bs + kPartStride;
        const float wb = mweight(bs[kHeadDim], bs[kHeadDim + 1], MB), wt = mweight(ts[kHeadDim], ts[kHeadDim + 1], MT);
        LB += wb * bs[kHeadDim + 1];
        OB = fmaf(wb, bs[tid], OB);
        LT += wt * ts[kHeadDim + 1];
        OT = fmaf(wt, ts[tid], OT);
      }
      const int64_t qp = qpos(p, b);
      if (decode) {
        // AS_{1:m-r}, normalised, with its ln-LSE: the rectified summary
        // the ring keeps for position m
        const float as = LB > 0.f ? OB * rcp_approx(LB) : 0.f;
        const float lse = LB > 0.f ? (MB + lg2_approx(LB)) * kLn2 : -INFINITY;
        const int64_t slot = (int64_t)bh * p.K + qp % p.K;
        if (p.app_o && len_ok(p, qp)) {
          p.app_o[slot * kHeadDim + tid] = as;
          if (tid == 0) {
            p.app_lse[slot] = lse;
            if (h == 0) p.app_pos[(int64_t)b * p.K + qp % p.K] = (int32_t)qp;
          }
        } else if (p.as_o) {
          p.as_o[(int64_t)bh * kHeadDim + tid] = as;
          if (tid == 0) p.as_lse[bh] = lse;
        }
        if (tid == 0 && p.match_pos_out) p.match_pos_out[bh] = pos;
      }
      // the output: AS with the tail (and the sink)
      const float M2 = fmaxf(LB > 0.f ? MB : -INFINITY, LT > 0.f ? MT : -INFINITY);
      const float wa = mweight(MB, LB, M2), wt = mweight(MT, LT, M2);
      const float L2 = wa * LB + wt * LT;
      p.out[(int64_t)bh * kHeadDim + tid] = L2 > 0.f ? (wa * OB + wt * OT) * rcp_approx(L2) : 0.f;
      if (tid == 0 && p.out_lse) p.out_lse[bh] = L2 > 0.f ? (M2 + lg2_approx(L2)) * kLn2 : -INFINITY;
    } else if (decode && tid < kHeadDim + kHeadDim / kPer) {
      // the step's query, for the ring (fused append) or the append kernel
      const int64_t qp = qpos(p, b);
      const int c = tid - kHeadDim;
      const uint4 qv = reinterpret_cast<const uint4 *>(p.q)[((int64_t)bh * p.q_stride + p.q_offset) / kPer + c];
      if (p.app_o && len_ok(p, qp))
        reinterpret_cast<uint4 *>(p.app_q)[((int64_t)bh * p.K + qp % p.K) * (kHeadDim / kPer) + c] = qv;
      else if (p.as_o)
        reinterpret_cast<uint4 *>(p.stage_q)[(int64_t)bh * (kHeadDim / kPer) + c] = qv;
    }
    block_sync();  // the combine area is free again
  }

  // The long bands: this CTA's span, piece by piece (one per unit it
  // meets); the CTA's warps take the piece's stages round-robin, then
  // combine their states into the piece's partial; pieces are counted per
  // unit (or per CTA group, whose last CTA merges the group).
  struct LongCur {
    int u, lo, hi, k;  // piece: unit, tokens [lo, hi]; the warp's next stage k (tokens lo + k * kStTok ..)
  };
  __device__ static bool piece_at(const StepParams &p, const Smem &S, int u, int64_t g0, int64_t g1, LongCur &C) {
    const int U = n_units(p);
#pragma unroll 1
    for (; u < U; ++u) {
      const int64_t a0 = S.off[u], z0 = S.off[u + 1];
      if (a0 >= g1) return false;
      const int64_t a = a0 > g0 ? a0 : g0, z = z0 < g1 ? z0 : g1;
      if (a < z) {
        C.u = u;
        C.lo = (int)(lb(p) + (a - a0));
        C.hi = (int)(lb(p) + (z - a0) - 1);
        return true;
      }
    }
    return false;
  }
  // the next stage of this warp from cursor C (kind -1: none left)
  __device__ static Desc long_next(const StepParams &p, const Smem &S, LongCur &C, int64_t g0, int64_t g1) {
    Desc d;
    d.kind = -1;
    d.u = d.a = d.cnt = 0;
#pragma unroll 1
    while (C.u >= 0) {
      const int a = C.lo + C.k * kStTok;
      if (a <= C.hi) {
        d.kind = 1;
        d.u = C.u;
        d.a = a;
        d.cnt = min(C.hi - a + 1, kStTok);
        C.k += kWarps;
        return d;
      }
      if (!piece_at(p, S, C.u + 1, g0, g1, C)) C.u = -1;
      C.k = warp_id();
    }
    return d;
  }

  // Merge of CTA group k of unit u's long band: its CTA pieces into the group
  // partial (the raw state).
  __device__ static void merge_group(const StepParams &p, int u, int c0, int c1, int k) {
    const int lane = lane_id(), hh = warp_id() / kWPH, wi = warp_id() % kWPH;
    const int dl = wi * kDW + min(lane, kLanes - 1) * kDL;
    const int a = max(c0, k * kGroupCtas), z = min(c1, k * kGroupCtas + kGroupCtas - 1);
    auto entry = [&](int i) -> const float * { return p.part_c + ((size_t)(u + a + i) * G + hh) * kPartStride; };
    Cls band, tail;
    merge_list(z - a + 1, z - a + 1, entry, dl, band, tail);
    float *dst = p.part_g + ((size_t)(u + k) * G + hh) * kPartStride;
    if (lane < kLanes) store_dims<kDL>(dst + dl, band.O);
    if (wi == 0 && lane == 0) *reinterpret_cast<float2 *>(dst + kHeadDim) = make_float2(band.M, band.L);
  }

  // The CTA's combine of its warps' states of a piece of unit u: part_x ->
  // part_c slot u + c, the warps in a fixed order.
  __device__ static void combine_warps(const StepParams &p, int u) {
    const int c = blockIdx.x;
    const float *x = p.part_x + (size_t)c * kWarps * G * kPartStride;
    float *dst = p.part_c + (size_t)(u + c) * G * kPartStride;
#pragma unroll 1
    for (int e = threadIdx.x; e < G * kHeadDim; e += kThreads) {
      const int hh = e / kHeadDim, dd = e % kHeadDim;
      float2 ml[kWarps];
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        ml[w] = __ldcg(reinterpret_cast<const float2 *>(x + (w * G + hh) * kPartStride + kHeadDim));
        if (ml[w].y > 0.f) M = fmaxf(M, ml[w].x);
      }
      float L = 0.f, O = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float wt = mweight(ml[w].x, ml[w].y, M);
        L += wt * ml[w].y;
        O = fmaf(wt, __ldcg(x + (w * G + hh) * kPartStride + dd), O);
      }
      dst[hh * kPartStride + dd] = O;
      if (dd == 0) *reinterpret_cast<float2 *>(dst + hh * kPartStride + kHeadDim) = make_float2(M, L);
    }
  }

  __device__ static void long_bands(const StepParams &p, const Smem &S, Ring &R) {
    const int c = blockIdx.x;
    if (c >= *S.Pl) return;
    const int64_t g0 = span(S, c), g1 = span(S, c + 1);
    LongCur F, C;  // fetch and consume cursors
    if (!piece_at(p, S, unit_of(p, S, g0), g0, g1, F)) return;
    F.k = warp_id();
    C = F;
    int32_t id[2];
    // prime
    Desc nx = long_next(p, S, F, g0, g1);
#pragma unroll 1
    for (int j = 0; j < kStages && nx.kind >= 0; ++j) {
      load_ids(p, nx, id);
      issue(p, R, nx, id);
      nx = long_next(p, S, F, g0, g1);
    }
    if (nx.kind >= 0) load_ids(p, nx, id);
    float2 q[G][kAPairs];
    Att A;
#pragma unroll 1
    while (C.u >= 0) {
      const int u = C.u;
      att_init(A);
      load_query(p, S, u, q);
#pragma unroll 1
      for (;;) {
        const int a = C.lo + C.k * kStTok;
        if (a > C.hi || *S.abort) break;
        const uint32_t n = R.used;
        if (wait_stage(p, S, R, n)) att_stage(A, q, stage_buf(R, n), a, R.rows[n % kStages], 1, 0x7fffffff);
        R.used++;
        C.k += kWarps;
        done_with_stage();
        if (nx.kind >= 0) {
          issue(p, R, nx, id);
          nx = long_next(p, S, F, g0, g1);
          if (nx.kind >= 0) load_ids(p, nx, id);
        }
      }
      att_finish(A, p.part_x + ((size_t)c * kWarps + warp_id()) * G * kPartStride);
      block_sync();  // the warp states are read back (from L2) by the other threads of the CTA
      combine_warps(p, u);
      block_sync();
      // count the piece: in its CTA group (two-level) or in the unit
      int c0, c1;
      long_run(S, u, &c0, &c1);
      const int k = c / kGroupCtas;
      if (threadIdx.x == 0) {
        int act = 0;
        if (grouped(c0, c1)) {
          const int a0 = max(c0, k * kGroupCtas), z0 = min(c1, k * kGroupCtas + kGroupCtas - 1);
          const uint32_t old = atom_add_acq_rel_u32(S.group_done + u + k, 1u);
          act = (int)old + 1 == z0 - a0 + 1 ? 1 : 0;
        } else {
          atom_add_acq_rel_u32(S.unit_done + u, 1u);
        }
        *S.flag = act;
      }
      block_sync();
      if (*S.flag) {
        // the last CTA of the group merges it, then counts it in the unit
        merge_group(p, u, c0, c1, k);
        block_sync();
        if (threadIdx.x == 0) {
          atom_add_acq_rel_u32(S.unit_done + u, 1u);
        }
      }
      // the next piece
      if (!piece_at(p, S, u + 1, g0, g1, C)) C.u = -1;
      C.k = warp_id();
    }
  }

  // Wait (bounded, thread 0 for the CTA) until a count reaches target.
  __device__ static void wait_count(const StepParams &p, const Smem &S, const uint32_t *ctr, uint32_t target) {
    if (threadIdx.x == 0) {
      const long long t0 = clock64();
      while (ld_acquire_u32(ctr) < target) {
        if (*S.abort) break;
        if (clock64() - t0 > p.wait_limit) {
          set_status(p.ctl, MAC_DEV_WAIT_TIMEOUT);
          *S.abort = 1;
          break;
        }
      }
    }
    block_sync();
  }
  // Wait until unit u's long-band entries are all in.
  __device__ static void wait_long(const StepParams &p, const Smem &S, int u) {
    int c0, c1;
    long_run(S, u, &c0, &c1);
    wait_count(p, S, S.unit_done + u, (uint32_t)long_entries(c0, c1));
  }

  // All CTAs of the (co-resident, cooperative) grid meet; bounded wait.
  __device__ static void grid_barrier(const StepParams &p, const Smem &S) {
    block_sync();
    if (threadIdx.x == 0) {
      unsigned long long *ctr = reinterpret_cast<unsigned long long *>(p.ctl + 2);
      const unsigned long long old = atom_add_release_u64(ctr, 1ull);
      const unsigned long long target = old - old % gridDim.x + gridDim.x;
      const long long t0 = clock64();
      while (ld_acquire_u64(ctr) < target) {
        if (clock64() - t0 > p.wait_limit) {
          set_status(p.ctl, MAC_DEV_WAIT_TIMEOUT);
          *S.abort = 1;
          break;
        }
      }
    }
    block_sync();
  }

  __device__ static void stamp(const StepParams &p, int k) {
    if (p.trace && threadIdx.x == 0) p.trace[(size_t)blockIdx.x * kTracePoints + k] = globaltimer();
  }

  // ---------------------------------------------------------------------

  __device__ static void run(const StepParams &p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_abort, s_par, s_Pl;
    __shared__ uint32_t s_flag;
    __shared__ int64_t s_T;
    __shared__ long long s_scan[kWarps];
    __shared__ int s_dec[kOwnMax];
    const int U = n_units(p), tid = threadIdx.x, w = warp_id();
    Smem S;
    S.stage = smem;
    S.full = reinterpret_cast<uint64_t *>(smem + kOffBar);
    S.rows = reinterpret_cast<int *>(smem + kOffMask);
    S.bd = reinterpret_cast<float *>(smem + kOffBd);
    S.off = reinterpret_cast<int64_t *>(smem + kOffUnits);
    S.um = reinterpret_cast<int32_t *>(S.off + U + 1);
    S.scan = s_scan;
    S.abort = &s_abort;
    S.ntok = &s_T;
    S.Pl = &s_Pl;
    S.flag = &s_flag;
    S.dec = s_dec;
    S.rope = p.B <= kRopeTab && p.rope_mode != MAC_ROPE_NONE ? reinterpret_cast<float2 *>(smem + off_rope(U)) : nullptr;
    S.pside = smem + off_pside(U, p.B);
    S.qbuf = p.qslot ? smem + off_qbuf(U, p.B) : nullptr;
    if (p.trace && tid == 0) p.trace[(size_t)blockIdx.x * kTracePoints + 16] = (unsigned long long)clock64();
    stamp(p, 0);
    if (tid < kWarps * kStages) mbar_init(smem_addr(&S.full[tid]), 1);
    if (tid == 0) {
      s_abort = 0;
      // decode launches alternate between the two buffers of minima
      s_par = (int)(*(volatile uint32_t *)(p.ctl + 6) & 1u);
    }
    mbar_fence_init();
    if (S.rope) {
      // the rotation angles of every request's query (shared by its heads)
#pragma unroll 1
      for (int i = tid; i < p.B * (kHeadDim / 2); i += kThreads) {
        const int b = i / (kHeadDim / 2), j = i % (kHeadDim / 2);
        float c, sn;
        rope_angle(qpos(p, b), p.rope_f[j], &c, &sn);
        S.rope[i] = make_float2(c, sn);
      }
    }
#pragma unroll 1
    for (int u = tid; u < U; u += kThreads) {
      const int64_t m = qpos(p, u / p.Hkv) - p.len_sub;
      const bool ok = len_ok(p, m);
      S.um[u] = ok ? (int32_t)m : 0;
      if (p.check_len && blockIdx.x == 0 && !ok) set_status(p.ctl, MAC_DEV_BAD_SEQ_LEN);
    }
    block_sync();
    S.best = p.best + (size_t)s_par * p.B * p.Hq;
    S.best_next = p.best + (size_t)(s_par ^ 1) * p.B * p.Hq;
    S.unit_done = p.unit_done + (size_t)s_par * U;
    S.unit_done_next = p.unit_done + (size_t)(s_par ^ 1) * U;
    S.group_done = p.group_done + (size_t)s_par * (U + kGroups);
    S.group_done_next = p.group_done + (size_t)(s_par ^ 1) * (U + kGroups);
    Ring R;
    R.buf = smem + (size_t)w * kStages * kStageBytes;
    R.bar0 = smem_addr(&S.full[w * kStages]);
    R.rows = S.rows + w * kStages;
    R.pside = S.pside + (size_t)w * kStages * kPosBytes;
    R.qbuf = S.qbuf ? S.qbuf + (size_t)w * 2 * kQE : nullptr;
    R.issued = R.used = 0;

    // owned heads, merged by this CTA
    const int NH = p.B * p.Hq;
    int h0, h_end, hstep;
    own_range(NH, &h0, &h_end, &hstep);
    const int nown = h_end > h0 ? (h_end - h0 + hstep - 1) / hstep : 0;
    const int nrnd = 1 + max(1, (nown + kWarps - 1) / kWarps);
    // round 0: phase A; round r >= 1: the boundary pieces of owned heads
    // (r-1) kWarps .. r kWarps - 1, then their merges.  One call site of the
    // streaming loop for all rounds.
#pragma unroll 1
    for (int rnd = 0; rnd < nrnd; ++rnd) {
      if (rnd == 1) {
        stamp(p, 1);
        grid_barrier(p, S);  // the minima of every head are final, the window tiles written
        stamp(p, 2);
        {
          // nobody reads the other buffers in this launch: clear them for the next
          const int i0 = blockIdx.x * kThreads + tid, di = gridDim.x * kThreads;
#pragma unroll 1
          for (int i = i0; i < p.B * p.Hq; i += di) S.best_next[i] = 0ull;
#pragma unroll 1
          for (int i = i0; i < U; i += di) S.unit_done_next[i] = 0u;
#pragma unroll 1
          for (int i = i0; i < U + kGroups; i += di) S.group_done_next[i] = 0u;
        }
        layout_long(p, S);
        stamp(p, 3);
      }
      if (*S.abort && rnd > 0) continue;
      stream(p, S, R, rnd, h0, hstep, nown);
      if (rnd > 0) {
        block_sync();  // the batch's boundary states are in S.bd
#pragma unroll 1
        for (int k = (rnd - 1) * kWarps; k < min(nown, rnd * kWarps) && !*S.abort; ++k)
          merge_one(p, S, h0 + k * hstep, false, k < kOwnMax ? S.dec[k] : -2, k - (rnd - 1) * kWarps);
      }
    }
    stamp(p, 4);
    if (!*S.abort) long_bands(p, S, R);
    stamp(p, 5);
#pragma unroll 1
    for (int bh = h0; bh < h_end; bh += hstep) {
      const int k = (bh - h0) / hstep;
      const int pos = k < kOwnMax ? S.dec[k] : decision(p, S, bh);
      const int u = (bh / p.Hq) * p.Hkv + (bh % p.Hq) / G;
      int c0, c1;
      long_run(S, u, &c0, &c1);
      if (c1 < c0 || pos >= 1 || *S.abort) continue;
      wait_long(p, S, u);
      if (*S.abort) continue;
      merge_one(p, S, bh, true, pos, 0);
    }
    stamp(p, 6);
    drain(p, R);
    block_sync();
    if (tid == 0) {
      // the last CTA to finish advances the launch count (which selects the
      // buffers of minima and counts the next launch uses)
      __threadfence();
      const uint32_t old = atomicAdd(p.ctl + 4, 1u);
      if (old == gridDim.x - 1) {
        p.ctl[4] = 0;
        atomicAdd(p.ctl + 6, 1u);
      }
      if (p.trace) {
        p.trace[(size_t)blockIdx.x * kTracePoints + 17] = (unsigned long long)clock64();
        p.trace[(size_t)blockIdx.x * kTracePoints + 7] = globaltimer();
      }
    }
  }
};

template <typename T, int G, bool PAGED>
__global__ void __launch_bounds__(kThreads, 1) step_kernel(const __grid_constant__ StepParams p) {
  Step<T, G, PAGED>::run(p);
}

}  // namespace ring
}  // namespace mac
