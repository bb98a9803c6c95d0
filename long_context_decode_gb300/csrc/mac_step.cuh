// mac_step.cuh -- one persistent kernel per decode step (cooperative launch,
// one CTA per SM).
//
//   Phase M (Match, [MAC] "Match (2)"/"Match (3)", K1): the pre-RoPE query
//   rings of all (request, head) pairs form one contiguous array of B*Hq*K
//   rows; CTA c streams rows [c*N/P, (c+1)*N/P) through shared memory and
//   computes each candidate's squared distance to its head's current query.
//   Each lane sums (a-b)^2 of its elements in a pairwise tree (a-b of two
//   bf16 values is exact in fp32) and the lanes of a row finish the tree with
//   shuffles, so the distance carries at most ~8 roundings; the pages'
//   expansion |a|^2+|b|^2-2a.b cancels badly for close pairs and is not
//   used.  A head's best (distance, position) is combined across CTAs with a
//   64-bit atomic max of a packed key, a total order (smaller distance, then
//   more recent position), so the result does not depend on scheduling.  The
//   last CTA to finish a (request, kv-head) unit turns the minima into
//   decisions and the unit's fresh-range start.
//
//   Tail chunks (Complete, K2, part 1): the last r tokens of every unit are
//   attended by every head whatever the match says (each head's band starts
//   at or before m-r+1), so they are streamed right after the match slice,
//   before the grid barrier.
//
//   Grid barrier; band chunks (K2, part 2): the band [s, m-r] of every unit,
//   which depends on the decisions, cut into chunks (plan_band) dealt
//   round-robin to the CTAs.  A GQA group loads each K/V tile once for its G
//   query heads ([MAC] "GQA intra-group skew"); heads that reuse from a later
//   position mask the tokens before their own band start.  Every chunk leaves
//   a partial summary (running max, sum, weighted values; base-2 log domain,
//   [MAC] "Complete").
//
//   Grid barrier; phase R: per (request, head), the chunk partials are merged
//   in a fixed order after the cached rectified summary of a hit head: the
//   band chunks give AS_{1:m-r}, the tail chunks then give the output.
//
// Full attention (and ring seeding) run the same attention code with s = 1,
// which is what makes a miss bitwise equal to it.  All phases stream through
// one ring of kStages shared-memory stages filled with 1-D TMA bulk copies
// (issued by thread 0, which polls the empty barriers without blocking and
// refills every stage it finds released) and drained by the CTA's 8 warps
// (full/empty mbarriers);
// every wait is bounded and reports MAC_DEV_WAIT_TIMEOUT instead of hanging.
#pragma once

#include "mac_common.cuh"

namespace mac {

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

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

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

template <typename T, int G, bool PAGED>
struct Step {
  static constexpr int kRowBytes = kHeadDim * (int)sizeof(T);
  static constexpr int kTileTok = kStageBytes / (2 * kRowBytes);  // 64 (bf16) / 32 (fp32)
  static constexpr int kTokPerGroup = kTileTok / 32;              // tokens per lane group per tile
  static constexpr int kMatchRows = kStageBytes / kRowBytes;      // ring rows per stage
  static constexpr int kPer = 16 / (int)sizeof(T);                // elements per 16-byte piece
  static constexpr int kNP = 16 / kPer;                           // pieces per lane (16 dims)
  static constexpr int kPairs = 8;                                // float2 pairs per lane (16 dims)
  static constexpr int kLPS = kHeadDim / kPer;                    // lanes per ring row
  static constexpr int kRowGroups = kThreads / kLPS;              // ring rows in flight per pass
  static constexpr int kQBytes = G * kRowBytes;

  // dynamic shared memory layout
  static constexpr size_t kOffQ = (size_t)kStages * kStageBytes;
  static constexpr size_t kOffBar = kOffQ + (size_t)kStages * kQBytes;
  static constexpr size_t kOffQrot = kOffBar + 128;
  static constexpr size_t kOffRed = kOffQrot + (size_t)G * kHeadDim * 4;
  static constexpr size_t kOffPos = kOffRed + (size_t)kWarps * G * kPartStride * 4;
  // phase M: ring positions of the requests a match slice touches; band
  // chunks and phase R: the first fresh token of every head
  static constexpr int kPosInts = kMaxHeads;
  static constexpr size_t kOffUnits = kOffPos + 4 * (size_t)kPosInts;
  // per unit: first band chunk (prefix, n_units + 1), query position, fresh-range start
  static size_t smem_bytes(int n_units) { return kOffUnits + 4 * (size_t)(3 * n_units + 1); }

  struct Smem {
    uint8_t *stage;     // [kStages][kStageBytes]
    uint8_t *qbuf;      // [kStages][kQBytes]
    uint64_t *full;     // [kStages]
    uint64_t *empty;    // [kStages]
    float *qrot;        // [G][d]
    float *red;         // [kWarps][G][kPartStride]
    int32_t *pos;       // [kPosInts]
    int32_t *prefix;    // [n_units + 1]
    int32_t *u_pos;     // [n_units]: position of the unit's query (RoPE angle pos - 1)
    int32_t *u_s;       // [n_units]: first token any head of the unit reads
    int *mask;          // [kStages]: valid 16-token pages of the tile in the stage
    volatile int *abort;
  };

  // Producer cursor, kept by thread 0: the next stage use to fill in the
  // CTA's sequence (match chunks, tail tiles, band tiles).  n counts the uses
  // issued so far; the consumers count the same sequence, so use n goes to
  // stage n % kStages.  Thread 0 never blocks on a release: it polls (pump)
  // after each of its own releases and while it waits for data.
  enum { P_MATCH = 0, P_TAIL = 1, P_IDLE = 2, P_BAND = 3, P_DONE = 4 };
  struct Producer {
    uint32_t n;
    int phase;
    int64_t r, s1;   // match: next ring row, end of the slice
    int item, total; // tail/band: current item index, number of items
    int k, ntiles, b, g, lo, hi;
    int64_t tile0;
  };

  // Lane `sub` (0..7) of a token's 8-lane group owns 16 dimensions: piece c
  // covers dims [c*8*kPer + sub*kPer, +kPer), so each group reads 128
  // contiguous bytes of a row per piece (no shared-memory bank conflicts).
  __device__ static int piece_dim(int c, int sub) { return c * 8 * kPer + sub * kPer; }

  // the scratch holds the chunk partials of lengths up to max_len only
  __device__ static bool len_ok(const StepParams &p, int64_t m) { return m >= 1 && m <= p.max_len; }
  __device__ static int64_t unit_len(const StepParams &p, const Smem &S, int u) {
    return (int64_t)S.u_pos[u] - p.len_sub;
  }

  __device__ static BandPlan plan(const StepParams &p, const Smem &S, int u) {
    const int64_t m = unit_len(p, S, u);
    if (!len_ok(p, m)) return plan_band(0, 1, p.r);
    return plan_band(m, S.u_s[u], p.r);
  }

  // tail chunk ti (unit ti / n_tail, chunk ti % n_tail)
  __device__ static void tail_item(const StepParams &p, const Smem &S, int ti, int *u, int *lo,
                                   int *hi) {
    *u = ti / p.n_tail;
    const int64_t m = unit_len(p, S, *u);
    int64_t a = 1, z = 0;
    if (len_ok(p, m)) tail_range(m, p.r, ti % p.n_tail, &a, &z);
    *lo = (int)a;
    *hi = (int)z;
  }

  __device__ static int unit_of_item(const int32_t *prefix, int n_units, int item) {
    int lo = 0, hi = n_units - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= item) lo = mid; else hi = mid - 1;
    }
    return lo;
  }

  // band chunk `item` (global index over all units' band chunks)
  __device__ static void band_item(const StepParams &p, const Smem &S, int item, int *u, int *lo,
                                   int *hi) {
    *u = unit_of_item(S.prefix, p.B * p.Hkv, item);
    int64_t a, z;
    band_range(plan(p, S, *u), p.r, item - S.prefix[*u], &a, &z);
    *lo = (int)a;
    *hi = (int)z;
  }

  // first CTA whose match slice contains ring row x
  __device__ static int cta_of_row(int64_t x, int64_t N, int P) {
    return (int)(((x + 1) * (int64_t)P - 1) / N);
  }

  // ---------------------------------------------------------------------
  // producer
  // ---------------------------------------------------------------------

  // Rows of K/V tile `tile` (tokens tile*kTileTok+1 .. +kTileTok) that fall in
  // [lo, hi], each copied to its own row of the stage, so no byte outside the
  // chunk is read; with_q also brings the unit's G pre-RoPE query rows.
  __device__ static void issue_tile(const StepParams &p, const Smem &S, int st, int b, int g, int lo,
                                    int hi, int64_t tile, bool with_q) {
    uint8_t *kbuf = S.stage + (size_t)st * kStageBytes;
    uint8_t *vbuf = kbuf + kStageBytes / 2;
    const uint32_t bar = smem_addr(&S.full[st]);
    const int64_t t0 = tile * kTileTok;
    uint32_t bytes = with_q ? (uint32_t)kQBytes : 0u;
    int msk = 0;
    int64_t ra[kTileTok / 16], rz[kTileTok / 16];
    int32_t pid[kTileTok / 16];
    if (!PAGED) {
      msk = (1 << (kTileTok / 16)) - 1;
      ra[0] = t0 + 1 > lo ? t0 + 1 : lo;
      rz[0] = t0 + kTileTok < hi ? t0 + kTileTok : hi;
      bytes += 2u * (uint32_t)(rz[0] - ra[0] + 1) * kRowBytes;
    } else {
      for (int pg = 0; pg < kTileTok / 16; ++pg) {
        const int64_t slot = tile * (kTileTok / 16) + pg;
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
        bytes += 2u * (uint32_t)(rz[pg] - ra[pg] + 1) * kRowBytes;
      }
    }
    S.mask[st] = msk;
    if (bytes == 0) {
      mbar_arrive(bar);
      return;
    }
    fence_proxy_async();
    mbar_expect_tx(bar, bytes);
    if (with_q) {
      const uint8_t *q = (const uint8_t *)p.q;
      for (int hh = 0; hh < G; ++hh) {
        const int64_t bh = (int64_t)b * p.Hq + g * G + hh;
        bulk_g2s(smem_addr(S.qbuf + (size_t)st * kQBytes + hh * kRowBytes),
                 q + (size_t)(bh * p.q_stride + p.q_offset) * sizeof(T), kRowBytes, bar);
      }
    }
    if (!PAGED) {
      const size_t off = (((size_t)b * p.Hkv + g) * (size_t)p.kv.capacity + (size_t)(ra[0] - 1)) * kRowBytes;
      const uint32_t n = (uint32_t)(rz[0] - ra[0] + 1) * kRowBytes;
      const uint32_t dst = (uint32_t)(ra[0] - t0 - 1) * kRowBytes;
      bulk_g2s(smem_addr(kbuf + dst), (const uint8_t *)p.kv.k + off, n, bar);
      bulk_g2s(smem_addr(vbuf + dst), (const uint8_t *)p.kv.v + off, n, bar);
    } else {
      for (int pg = 0; pg < kTileTok / 16; ++pg) {
        if (pid[pg] < 0) continue;
        const size_t off = (((size_t)pid[pg] * p.Hkv + g) * 16 + (size_t)((ra[pg] - 1) % 16)) * kRowBytes;
        const uint32_t n = (uint32_t)(rz[pg] - ra[pg] + 1) * kRowBytes;
        const uint32_t dst = (uint32_t)(ra[pg] - t0 - 1) * kRowBytes;
        bulk_g2s(smem_addr(kbuf + dst), (const uint8_t *)p.kv.k + off, n, bar);
        bulk_g2s(smem_addr(vbuf + dst), (const uint8_t *)p.kv.v + off, n, bar);
      }
    }
  }

  // next chunk of the match slice: rows [r, e) within one head, <= kMatchRows
  __device__ static int64_t chunk_end(int64_t r, int64_t s1, int K) {
    int64_t e = r + kMatchRows;
    const int64_t head_end = (r / K + 1) * K;
    if (e > head_end) e = head_end;
    if (e > s1) e = s1;
    return e;
  }

  // Position the cursor on the next stage use of the CTA's sequence; false
  // when the current phase has nothing more (tail -> idle until the band
  // chunks are known, band -> done).
  __device__ static bool next_use(const StepParams &p, const Smem &S, Producer &pr) {
    for (;;) {
      if (pr.phase == P_MATCH) {
        if (pr.r < pr.s1) return true;
        pr.phase = P_TAIL;
        pr.item = -1;
        pr.total = p.B * p.Hkv * p.n_tail;
        pr.k = pr.ntiles = 0;
      }
      if (pr.phase != P_TAIL && pr.phase != P_BAND) return false;
      if (pr.k < pr.ntiles) return true;
      pr.item = pr.item < 0 ? (int)blockIdx.x : pr.item + (int)gridDim.x;
      if (pr.item >= pr.total) {
        pr.phase = pr.phase == P_TAIL ? P_IDLE : P_DONE;
        return false;
      }
      int u;
      if (pr.phase == P_TAIL)
        tail_item(p, S, pr.item, &u, &pr.lo, &pr.hi);
      else
        band_item(p, S, pr.item, &u, &pr.lo, &pr.hi);
      pr.b = u / p.Hkv;
      pr.g = u % p.Hkv;
      pr.k = 0;
      pr.ntiles = 0;
      if (pr.lo <= pr.hi) {
        pr.tile0 = (pr.lo - 1) / kTileTok;
        pr.ntiles = (int)((pr.hi - 1) / kTileTok - pr.tile0 + 1);
      }
    }
  }

  // Issue the use the cursor is on into stage pr.n % kStages (free) and advance.
  __device__ static void issue_current(const StepParams &p, const Smem &S, Producer &pr) {
    const int st = pr.n % kStages;
    if (pr.phase == P_MATCH) {
      const int64_t e = chunk_end(pr.r, pr.s1, p.K);
      if (!*S.abort) {
        const uint32_t bytes = (uint32_t)(e - pr.r) * kRowBytes;
        const uint32_t bar = smem_addr(&S.full[st]);
        fence_proxy_async();
        mbar_expect_tx(bar, bytes);
        bulk_g2s(smem_addr(S.stage + (size_t)st * kStageBytes),
                 (const uint8_t *)p.ring_q + (size_t)pr.r * kRowBytes, bytes, bar);
      }
      pr.r = e;
    } else {
      if (!*S.abort) issue_tile(p, S, st, pr.b, pr.g, pr.lo, pr.hi, pr.tile0 + pr.k, pr.k == 0);
      ++pr.k;
    }
    ++pr.n;
  }

  // Issue every next use whose stage is already free, without blocking
  // (thread 0 only).  Thread 0 also consumes tiles, so it must never wait
  // for the other warps here: it refills as soon as it finds a stage free,
  // here after each of its own releases and inside its own waits.
  __device__ static void pump(const StepParams &p, const Smem &S, Producer &pr) {
    while (next_use(p, S, pr)) {
      const int st = pr.n % kStages;
      if (!*S.abort &&
          !mbar_test_wait(smem_addr(&S.empty[st]), ((pr.n / kStages) & 1u) ^ 1u))
        return;
      issue_current(p, S, pr);
    }
  }

  // Consumer wait for stage use n; thread 0 keeps the copies flowing while
  // it waits.  Bounded like every wait (about a second, or at once after an
  // abort).
  __device__ static bool wait_full_pump(const StepParams &p, const Smem &S, Producer &pr, int st,
                                        uint32_t n) {
    const uint32_t bar = smem_addr(&S.full[st]);
    const uint32_t parity = n & 1u;
    if (threadIdx.x != 0) return mbar_wait_bounded(bar, parity, S.abort);
    const long long t0 = clock64();
    for (;;) {
      if (mbar_test_wait(bar, parity)) return true;
      pump(p, S, pr);
      if (*S.abort || clock64() - t0 > (1LL << 31)) return false;
    }
  }

  // ---------------------------------------------------------------------
  // phase M
  // ---------------------------------------------------------------------

  // Combine the CTA's running best of head bh and publish it.
  __device__ static void flush_best(const StepParams &p, int64_t bh, float bd, int bp, float *s_bd,
                                    int *s_bp) {
    const int ct = threadIdx.x, warp = ct >> 5, lane = ct & 31;
#pragma unroll
    for (int off = 16; off >= kLPS; off >>= 1) {
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
    consumer_sync();
    if (ct == 0) {
      for (int w = 1; w < kWarps; ++w)
        if (better(s_bd[w], s_bp[w], bd, bp)) {
          bd = s_bd[w];
          bp = s_bp[w];
        }
      if (bp >= 1) atomicMax(&p.best[bh], pack_best(bd, bp));
    }
    consumer_sync();
  }

  // Decisions of unit u from the combined minima ([MAC] K1: hit iff the
  // smallest squared distance is strictly below thr^2).
  __device__ static void finalize_unit(const StepParams &p, int u) {
    const int b = u / p.Hkv, g = u % p.Hkv;
    const int64_t m = (int64_t)p.pos_base[b] + p.pos_add - p.len_sub;
    const bool m_ok = len_ok(p, m);
    if (!m_ok && p.check_len) set_status(p.ctl, MAC_DEV_BAD_SEQ_LEN);
    int s = 0x7fffffff;
    for (int hh = 0; hh < G; ++hh) {
      const int64_t bh = (int64_t)b * p.Hq + g * G + hh;
      const unsigned long long inv = atomicExch(&p.best[bh], 0ull);
      bool hit = false;
      int pos = -1;
      if (inv != 0ull) {
        const unsigned long long key = ~inv;
        const float d = __uint_as_float((uint32_t)(key >> 32));
        pos = (int)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
        hit = m_ok && d < p.thr2 && m >= p.min_context;
      }
      const int lo = hit ? (pos - p.r + 1 > 1 ? pos - p.r + 1 : 1) : 1;
      p.head_info[bh] = make_int2(hit ? pos : -1, lo);
      if (p.match_pos_out) p.match_pos_out[bh] = hit ? pos : -1;
      s = lo < s ? lo : s;
    }
    p.unit_s[u] = s;
    p.match_cnt[u] = 0;
  }

  __device__ static void match_phase(const StepParams &p, const Smem &S, uint32_t &tc, Producer &pr) {
    __shared__ float s_bd[kWarps];
    __shared__ int s_bp[kWarps];
    const int64_t N = (int64_t)p.B * p.Hq * p.K;
    const int P = gridDim.x, c = blockIdx.x;
    const int64_t s0 = (int64_t)c * N / P, s1 = (int64_t)(c + 1) * N / P;
    const int ct = threadIdx.x, lane = ct & 31;
    const int sub = lane % kLPS;  // lane within its row
    const int rg = ct / kLPS;     // row group (rows rg, rg + kRowGroups, ...)
    const unsigned gmask = kLPS == 32 ? 0xffffffffu : (0xffffu << (lane & 16));

    // slot positions of the requests the slice touches, staged in shared
    // memory once (they are shared by all heads of a request)
    const int64_t rows_per_req = (int64_t)p.Hq * p.K;
    const int b_lo = (int)(s0 / rows_per_req);
    const int b_hi = s1 > s0 ? (int)((s1 - 1) / rows_per_req) : b_lo - 1;
    const bool staged = (int64_t)(b_hi - b_lo + 1) * p.K <= kPosInts;
    if (staged) {
      const int n = (b_hi - b_lo + 1) * p.K;
      const int32_t *src = p.ring_pos + (int64_t)b_lo * p.K;
      for (int i = ct; i < n; i += kThreads) S.pos[i] = src[i];
    }
    __syncthreads();

    int64_t cur = -1;
    float bd = INFINITY;
    int bp = -1;
    float2 qv[kPer / 2];
    int pos_lo = 1, pos_hi = 0;
    const int32_t *rpos = p.ring_pos;
    for (int64_t r = s0; r < s1;) {
      const int64_t e = chunk_end(r, s1, p.K);
      const int64_t bh = r / p.K;
      const int b = (int)(bh / p.Hq);
      if (bh != cur) {
        if (cur >= 0) flush_best(p, cur, bd, bp, s_bd, s_bp);
        cur = bh;
        bd = INFINITY;
        bp = -1;
        unpack16x2<T>(reinterpret_cast<const uint4 *>(p.q)[(bh * p.q_stride + p.q_offset) / kPer + sub], qv);
        const int64_t m = (int64_t)S.u_pos[b * p.Hkv] - p.len_sub;
        if (len_ok(p, m)) {
          pos_lo = m - p.K > 1 ? (int)(m - p.K) : 1;
          pos_hi = (int)(m - 1);
        } else {
          pos_lo = 1;
          pos_hi = 0;
        }
        rpos = staged ? S.pos + (int64_t)(b - b_lo) * p.K : p.ring_pos + (int64_t)b * p.K;
      }
      const int st = tc % kStages;
      const bool ok = wait_full_pump(p, S, pr, st, tc / kStages);
      if (!ok) *S.abort = 1;
      const int n = (int)(e - r);
      const int slot0 = (int)(r % p.K);
      const uint8_t *rows = S.stage + (size_t)st * kStageBytes;
      for (int i = rg; i < n; i += kRowGroups) {
        const uint4 v = *reinterpret_cast<const uint4 *>(rows + (size_t)i * kRowBytes + sub * 16);
        const int ps = rpos[slot0 + i];
        float2 e2[kPer / 2];
        unpack16x2<T>(v, e2);
        // squared differences, then a pairwise tree: element k of the lane's
        // piece is added to element k + kPer/2, k + kPer/4, ... (the packed
        // pairs hold elements (2i, 2i+1), so each level adds pair i to pair
        // i + w2/2 and the last level adds the two halves of a pair)
#pragma unroll
        for (int k = 0; k < kPer / 2; ++k) {
          const float2 df = __fadd2_rn(qv[k], make_float2(-e2[k].x, -e2[k].y));  // exact for bf16
          e2[k] = __fmul2_rn(df, df);
        }
#pragma unroll
        for (int w2 = kPer / 4; w2 >= 1; w2 >>= 1)
#pragma unroll
          for (int k = 0; k < w2; ++k) e2[k] = __fadd2_rn(e2[k], e2[k + w2]);
        float D = __fadd_rn(e2[0].x, e2[0].y);
#pragma unroll
        for (int off = kLPS / 2; off >= 1; off >>= 1)
          D = __fadd_rn(D, __shfl_xor_sync(gmask, D, off));
        if (ok && ps >= pos_lo && ps <= pos_hi && better(D, ps, bd, bp)) {
          bd = D;
          bp = ps;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&S.empty[st]));
      if (ct == 0) pump(p, S, pr);
      ++tc;
      r = e;
    }
    if (cur >= 0) flush_best(p, cur, bd, bp, s_bd, s_bp);

    // count this CTA off every unit its slice touched; the last one decides
    if (ct == 0 && s0 < s1) {
      const int64_t rows_per_unit = (int64_t)G * p.K;
      const int u0 = (int)(s0 / rows_per_unit), u1 = (int)((s1 - 1) / rows_per_unit);
      __threadfence();
      for (int u = u0; u <= u1; ++u) {
        // CTAs whose (non-empty) slice meets the unit: with N >= P every
        // slice holds >= 1 row, so all CTAs from the one holding the unit's
        // first row to the one holding its last; with N < P every non-empty
        // slice holds exactly one row, one CTA per row of the unit
        const int first = cta_of_row((int64_t)u * rows_per_unit, N, P);
        const int last = cta_of_row((int64_t)(u + 1) * rows_per_unit - 1, N, P);
        const int64_t target = N >= P ? (int64_t)(last - first + 1) : rows_per_unit;
        if (atomicAdd(&p.match_cnt[u], 1) == target - 1) {
          __threadfence();
          finalize_unit(p, u);
        }
      }
    }
  }

  // All CTAs of the (co-resident, cooperative) grid meet; bounded wait.
  __device__ static void grid_barrier(const StepParams &p, const Smem &S) {
    if (threadIdx.x == 0) {
      unsigned long long *ctr = reinterpret_cast<unsigned long long *>(p.ctl + 2);
      __threadfence();
      const unsigned long long old = atomicAdd(ctr, 1ull);
      const unsigned long long target = old - old % gridDim.x + gridDim.x;
      const long long t0 = clock64();
      while (ld_acquire_u64(ctr) < target) {
        if (clock64() - t0 > (1LL << 31)) {
          set_status(p.ctl, MAC_DEV_WAIT_TIMEOUT);
          *S.abort = 1;
          break;
        }
        __nanosleep(32);
      }
      __threadfence();
    }
    __syncthreads();
  }

  // ---------------------------------------------------------------------
  // attention over one chunk
  // ---------------------------------------------------------------------

  // Attend the unit's G heads to tokens [lo, hi] (heads with lo_h > t skip
  // token t) and store the chunk's partial summaries at dst.
  __device__ static void process_chunk(const StepParams &p, const Smem &S, uint32_t &tc,
                                       Producer &pr, int u, int lo, int hi, const int *lo_h,
                                       float *dst) {
    const int ct = threadIdx.x, warp = ct >> 5, lane = ct & 31;
    const int lg = lane >> 3, sub = lane & 7;
    float2 q[G][kPairs], o[G][kPairs];
    float mrun[G], lrun[G];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      mrun[hh] = -INFINITY;
      lrun[hh] = 0.f;
#pragma unroll
      for (int i = 0; i < kPairs; ++i) o[hh][i] = make_float2(0.f, 0.f);
    }

    if (lo <= hi) {
      const int64_t tile0 = (lo - 1) / kTileTok;
      const int ntiles = (int)((hi - 1) / kTileTok - tile0 + 1);
      for (int k = 0; k < ntiles; ++k) {
        const int st = tc % kStages;
        const bool ok = wait_full_pump(p, S, pr, st, tc / kStages);
        if (!ok) *S.abort = 1;
        if (k == 0) {
          // R(pos) q~ * log2(e)/sqrt(d) for the unit's heads, from the query
          // rows that came with the first tile
          const int64_t pos = S.u_pos[u];
          for (int idx = ct; idx < G * (kHeadDim / 2); idx += kThreads) {
            const int hh = idx / (kHeadDim / 2), j = idx % (kHeadDim / 2);
            if (!rope_rotate_pair<T>(S.qbuf + (size_t)st * kQBytes, (int64_t)hh * kHeadDim,
                                     S.qrot + hh * kHeadDim, j, pos, p.rope_mode, p.rope_w[j],
                                     p.q_scale))
              set_status(p.ctl, MAC_DEV_NONFINITE_Q);
          }
          consumer_sync();
#pragma unroll
          for (int hh = 0; hh < G; ++hh)
#pragma unroll
            for (int c = 0; c < kNP; ++c)
#pragma unroll
              for (int e4 = 0; e4 < kPer; e4 += 4) {
                const float4 v =
                    *reinterpret_cast<const float4 *>(S.qrot + hh * kHeadDim + piece_dim(c, sub) + e4);
                q[hh][(c * kPer + e4) / 2] = make_float2(v.x, v.y);
                q[hh][(c * kPer + e4) / 2 + 1] = make_float2(v.z, v.w);
              }
        }
        const uint8_t *kb = S.stage + (size_t)st * kStageBytes;
        const uint8_t *vb = kb + kStageBytes / 2;
        const int t0 = (int)((tile0 + k) * kTileTok);
        const int msk = S.mask[st];
        float sc[kTokPerGroup][G];
        bool tv[kTokPerGroup];
#pragma unroll
        for (int j = 0; j < kTokPerGroup; ++j) {
          const int row = j * 32 + warp * 4 + lg;
          const int t = t0 + row + 1;
          tv[j] = ok && t >= lo && t <= hi && ((msk >> (row >> 4)) & 1);
          float2 kf[kPairs];
#pragma unroll
          for (int c = 0; c < kNP; ++c)
            unpack16x2<T>(*reinterpret_cast<const uint4 *>(kb + row * kRowBytes + c * 128 + sub * 16),
                          kf + c * (kPer / 2));
#pragma unroll
          for (int hh = 0; hh < G; ++hh) {
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < kPairs; ++i) acc = __ffma2_rn(q[hh][i], kf[i], acc);
            float a = acc.x + acc.y;
            a += __shfl_xor_sync(0xffffffffu, a, 1);
            a += __shfl_xor_sync(0xffffffffu, a, 2);
            a += __shfl_xor_sync(0xffffffffu, a, 4);
            sc[j][hh] = a;
          }
        }
        // one rescale per head per tile, then accumulate the tile's tokens
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          float mx = -INFINITY;
#pragma unroll
          for (int j = 0; j < kTokPerGroup; ++j) {
            const int t = t0 + j * 32 + warp * 4 + lg + 1;
            if (tv[j] && t >= lo_h[hh]) mx = fmaxf(mx, sc[j][hh]);
          }
          if (mx > mrun[hh]) {
            const float f = ex2(mrun[hh] - mx);
            const float2 f2 = make_float2(f, f);
            lrun[hh] *= f;
#pragma unroll
            for (int i = 0; i < kPairs; ++i) o[hh][i] = __fmul2_rn(o[hh][i], f2);
            mrun[hh] = mx;
          }
        }
#pragma unroll
        for (int j = 0; j < kTokPerGroup; ++j) {
          const int row = j * 32 + warp * 4 + lg;
          const int t = t0 + row + 1;
          float2 vf[kPairs];
#pragma unroll
          for (int c = 0; c < kNP; ++c)
            unpack16x2<T>(*reinterpret_cast<const uint4 *>(vb + row * kRowBytes + c * 128 + sub * 16),
                          vf + c * (kPer / 2));
#pragma unroll
          for (int hh = 0; hh < G; ++hh) {
            if (tv[j] && t >= lo_h[hh]) {
              const float w = ex2(sc[j][hh] - mrun[hh]);
              const float2 w2 = make_float2(w, w);
              lrun[hh] += w;
#pragma unroll
              for (int i = 0; i < kPairs; ++i) o[hh][i] = __ffma2_rn(w2, vf[i], o[hh][i]);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&S.empty[st]));
        if (ct == 0) pump(p, S, pr);
        ++tc;
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
        const float2 a2 = make_float2(a, a), cc = make_float2(c2, c2);
#pragma unroll
        for (int i = 0; i < kPairs; ++i) {
          const float2 other = make_float2(__shfl_xor_sync(0xffffffffu, o[hh][i].x, off),
                                           __shfl_xor_sync(0xffffffffu, o[hh][i].y, off));
          o[hh][i] = __ffma2_rn(other, cc, __fmul2_rn(o[hh][i], a2));
        }
        mrun[hh] = lrun[hh] > 0.f ? mn : -INFINITY;
      }
    }
    if (lg == 0) {
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        float *rw = S.red + ((size_t)warp * G + hh) * kPartStride;
#pragma unroll
        for (int c = 0; c < kNP; ++c)
#pragma unroll
          for (int e = 0; e < kPer; e += 2) {
            const float2 v = o[hh][(c * kPer + e) / 2];
            rw[piece_dim(c, sub) + e] = v.x;
            rw[piece_dim(c, sub) + e + 1] = v.y;
          }
        if (sub == 0) {
          rw[kHeadDim] = mrun[hh];
          rw[kHeadDim + 1] = lrun[hh];
        }
      }
    }
    consumer_sync();
    // the warps in a fixed order -> the chunk's partial
    for (int idx = ct; idx < G * kHeadDim; idx += kThreads) {
      const int hh = idx / kHeadDim, dim = idx % kHeadDim;
      float M = -INFINITY, L = 0.f, O = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float *rw = S.red + ((size_t)w * G + hh) * kPartStride;
        const float m2 = rw[kHeadDim], l2 = rw[kHeadDim + 1], o2 = rw[dim];
        if (l2 == 0.f) continue;
        if (L == 0.f) {
          M = m2;
          L = l2;
          O = o2;
          continue;
        }
        const float mn = fmaxf(M, m2);
        const float a = ex2(M - mn), c2 = ex2(m2 - mn);
        L = L * a + l2 * c2;
        O = O * a + o2 * c2;
        M = mn;
      }
      float *out = dst + (size_t)hh * kPartStride;
      out[dim] = O;
      if (dim == 0) {
        out[kHeadDim] = M;
        out[kHeadDim + 1] = L;
      }
    }
    consumer_sync();  // S.red is rewritten by the next chunk
  }

  // ---------------------------------------------------------------------
  // layout of the band chunks (after the match)
  // ---------------------------------------------------------------------

  // Cache every unit's fresh-range start and every head's first fresh token
  // in shared memory, then lay the band chunks out: prefix[u] = first band
  // chunk of unit u, prefix[n_units] = total.
  __device__ static void build_prefix(const StepParams &p, const Smem &S, int n_units) {
    __shared__ int wsum[kWarps];
    int32_t *prefix = S.prefix;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int bh = tid; bh < p.B * p.Hq; bh += kThreads)
      S.pos[bh] = p.mode == MODE_DECODE ? __ldcg(&p.head_info[bh]).y : 1;
    const int seg = (n_units + kThreads - 1) / kThreads;
    const int beg = tid * seg;
    const int end = min(beg + seg, n_units);
    for (int u = beg; u < end; ++u) S.u_s[u] = p.mode == MODE_DECODE ? __ldcg(&p.unit_s[u]) : 1;
    int run = 0;
    for (int u = beg; u < end; ++u) {
      run += plan(p, S, u).nb;
      prefix[u + 1] = run;
    }
    int x = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = lane < kWarps ? wsum[lane] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, off);
        if (lane >= off) w += y;
      }
      if (lane < kWarps) wsum[lane] = w;
    }
    __syncthreads();
    const int excl = x - run + (warp > 0 ? wsum[warp - 1] : 0);
    for (int u = beg; u < end; ++u) prefix[u + 1] += excl;
    if (tid == 0) prefix[0] = 0;
    __syncthreads();
  }

  // ---------------------------------------------------------------------
  // phase R
  // ---------------------------------------------------------------------

  // (M, L, O[4]) <- (M, L, O) (+) (m2, l2, o2[4]) in base-2 log domain; an
  // empty operand (L == 0) is the identity.
  __device__ static void merge4(float &M, float &L, float *O, float m2, float l2, const float *o2) {
    if (l2 == 0.f) return;
    if (L == 0.f) {
      M = m2;
      L = l2;
#pragma unroll
      for (int i = 0; i < 4; ++i) O[i] = o2[i];
      return;
    }
    const float mn = fmaxf(M, m2);
    const float a = ex2(M - mn), c = ex2(m2 - mn);
    L = L * a + l2 * c;
#pragma unroll
    for (int i = 0; i < 4; ++i) O[i] = O[i] * a + o2[i] * c;
    M = mn;
  }

  // For each (request, head) -- one per CTA at a time -- merge the unit's
  // chunk partials in order: band chunks, then tail chunks.  The 8 warps
  // each take a contiguous segment of that list (lane l owns dims 4l..4l+3)
  // and keep two running states, band and tail.  Warp 0 then merges, in
  // order: the cached summary of a hit head, the band states of warps 0..7
  // (giving AS_{1:m-r}), and the tail states (giving the output).
  __device__ static void reduce_phase(const StepParams &p, const Smem &S) {
    constexpr int kSeg = kHeadDim + 4;                // m, l, -, -, o[d]
    float *seg = reinterpret_cast<float *>(S.stage);  // [kWarps][2][kSeg]; the stages are idle now
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_bh = p.B * p.Hq;
    for (int bh = blockIdx.x; bh < n_bh; bh += gridDim.x) {
      const int b = bh / p.Hq, h = bh % p.Hq, g = h / G, hh = h % G;
      const int u = b * p.Hkv + g;
      const int first = S.prefix[u];
      const int nb = S.prefix[u + 1] - first;
      const int n = nb + p.n_tail;
      if (p.mode == MODE_DECODE && warp == kWarps - 1 && lane < kHeadDim / kPer) {
        // the append (on the aux stream) reads the step's query from the ring
        // workspace, so the caller may reuse its query buffer right away
        reinterpret_cast<uint4 *>(p.stage_q)[(int64_t)bh * (kHeadDim / kPer) + lane] =
            reinterpret_cast<const uint4 *>(p.q)[((int64_t)bh * p.q_stride + p.q_offset) / kPer + lane];
      }
      const int per = (n + kWarps - 1) / kWarps;
      const int i0 = warp * per, i1 = min(n, i0 + per);
      float bm = -INFINITY, bl = 0.f, bo[4] = {0.f, 0.f, 0.f, 0.f};
      float tm = -INFINITY, tl = 0.f, to[4] = {0.f, 0.f, 0.f, 0.f};
      for (int i = i0; i < i1; i += 4) {
        float pm[4], pl[4], po[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (i + j < i1) {
            const int it = i + j;
            const float *pp = it < nb ? p.partials + ((int64_t)(first + it) * G + hh) * kPartStride
                                      : p.tail_part + (((int64_t)u * p.n_tail + (it - nb)) * G + hh) * kPartStride;
            pm[j] = __ldcg(pp + kHeadDim);
            pl[j] = __ldcg(pp + kHeadDim + 1);
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(pp) + lane);
            po[j][0] = v.x;
            po[j][1] = v.y;
            po[j][2] = v.z;
            po[j][3] = v.w;
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (i + j >= i1) break;
          if (i + j < nb)
            merge4(bm, bl, bo, pm[j], pl[j], po[j]);
          else
            merge4(tm, tl, to, pm[j], pl[j], po[j]);
        }
      }
      float *sw = seg + (size_t)warp * 2 * kSeg;
      if (lane == 0) {
        sw[0] = bm;
        sw[1] = bl;
        sw[kSeg] = tm;
        sw[kSeg + 1] = tl;
      }
      *reinterpret_cast<float4 *>(sw + 4 + lane * 4) = make_float4(bo[0], bo[1], bo[2], bo[3]);
      *reinterpret_cast<float4 *>(sw + kSeg + 4 + lane * 4) = make_float4(to[0], to[1], to[2], to[3]);
      __syncthreads();
      if (warp == 0) {
        float M = -INFINITY, L = 0.f, O[4] = {0.f, 0.f, 0.f, 0.f};
        if (p.mode == MODE_DECODE) {
          const int2 hi = __ldcg(&p.head_info[bh]);
          if (hi.x >= 1) {
            const int64_t slot = (int64_t)bh * p.K + hi.x % p.K;
            const float lse = p.ring_lse[slot];
            if (lse > -INFINITY) {
              const float4 v = reinterpret_cast<const float4 *>(p.ring_o + slot * kHeadDim)[lane];
              const float a[4] = {v.x, v.y, v.z, v.w};
              merge4(M, L, O, lse * kLog2e, 1.f, a);
            }
          }
        }
        for (int w = 0; w < kWarps; ++w) {
          const float *s = seg + (size_t)w * 2 * kSeg;
          merge4(M, L, O, s[0], s[1], s + 4 + lane * 4);
        }
        if (p.as_o) {
          const float inv = L > 0.f ? 1.f / L : 0.f;
          *reinterpret_cast<float4 *>(p.as_o + (int64_t)bh * kHeadDim + lane * 4) =
              make_float4(O[0] * inv, O[1] * inv, O[2] * inv, O[3] * inv);
          if (lane == 0) p.as_lse[bh] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
        }
        for (int w = 0; w < kWarps; ++w) {
          const float *s = seg + (size_t)w * 2 * kSeg + kSeg;
          merge4(M, L, O, s[0], s[1], s + 4 + lane * 4);
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        *reinterpret_cast<float4 *>(p.out + (int64_t)bh * kHeadDim + lane * 4) =
            make_float4(O[0] * inv, O[1] * inv, O[2] * inv, O[3] * inv);
        if (p.out_lse && lane == 0) p.out_lse[bh] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
      }
      __syncthreads();
    }
  }

  // ---------------------------------------------------------------------

  __device__ static void run(const StepParams &p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_mask[kStages];
    __shared__ int s_abort;
    const int n_units = p.B * p.Hkv;
    Smem S;
    S.stage = smem;
    S.qbuf = smem + kOffQ;
    S.full = reinterpret_cast<uint64_t *>(smem + kOffBar);
    S.empty = S.full + kStages;
    S.qrot = reinterpret_cast<float *>(smem + kOffQrot);
    S.red = reinterpret_cast<float *>(smem + kOffRed);
    S.pos = reinterpret_cast<int32_t *>(smem + kOffPos);
    S.prefix = reinterpret_cast<int32_t *>(smem + kOffUnits);
    S.u_pos = S.prefix + (n_units + 1);
    S.u_s = S.u_pos + n_units;
    S.mask = s_mask;
    S.abort = &s_abort;

    const int tid = threadIdx.x;
    unsigned long long *trace = p.trace ? p.trace + (size_t)blockIdx.x * kTracePoints : nullptr;
    if (trace && tid == 0) trace[0] = globaltimer();
    if (tid == 0) {
      for (int i = 0; i < kStages; ++i) {
        mbar_init(smem_addr(&S.full[i]), 1);
        mbar_init(smem_addr(&S.empty[i]), kWarps);
      }
      s_abort = 0;
      mbar_fence_init();
    }
    for (int u = tid; u < n_units; u += kThreads)
      S.u_pos[u] = (int32_t)((int64_t)p.pos_base[u / p.Hkv] + p.pos_add);
    __syncthreads();

    uint32_t tc = 0;  // stage uses consumed so far (every thread counts the same sequence)
    Producer pr;      // meaningful in thread 0 only
    if (tid == 0) {
      const int64_t N = (int64_t)p.B * p.Hq * p.K;
      pr.n = 0;
      pr.phase = p.mode == MODE_DECODE ? P_MATCH : P_TAIL;
      pr.r = (int64_t)blockIdx.x * N / gridDim.x;
      pr.s1 = p.mode == MODE_DECODE ? (int64_t)(blockIdx.x + 1) * N / gridDim.x : pr.r;
      pr.item = -1;
      pr.total = n_units * p.n_tail;
      pr.k = pr.ntiles = 0;
      pump(p, S, pr);
    }

    if (p.mode == MODE_DECODE) match_phase(p, S, tc, pr);
    if (trace && tid == 0) trace[1] = globaltimer();
    // tail chunks: independent of the match
    const int all1[4] = {1, 1, 1, 1};
    for (int ti = blockIdx.x; ti < n_units * p.n_tail; ti += gridDim.x) {
      int u, lo, hi;
      tail_item(p, S, ti, &u, &lo, &hi);
      process_chunk(p, S, tc, pr, u, lo, hi, all1,
                    p.tail_part + (size_t)ti * G * kPartStride);
    }
    __syncthreads();
    if (trace && tid == 0) trace[2] = globaltimer();
    if (p.mode == MODE_DECODE) grid_barrier(p, S);  // decisions and unit starts are visible
    if (trace && tid == 0) trace[3] = globaltimer();

    build_prefix(p, S, n_units);
    const int total = S.prefix[n_units];
    if (tid == 0) {
      pr.phase = P_BAND;
      pr.item = -1;
      pr.total = total;
      pr.k = pr.ntiles = 0;
      pump(p, S, pr);
    }
    for (int item = blockIdx.x; item < total; item += gridDim.x) {
      int u, lo, hi;
      band_item(p, S, item, &u, &lo, &hi);
      const int b = u / p.Hkv, g = u % p.Hkv;
      int lo_h[G];
#pragma unroll
      for (int hh = 0; hh < G; ++hh) lo_h[hh] = S.pos[b * p.Hq + g * G + hh];
      process_chunk(p, S, tc, pr, u, lo, hi, lo_h, p.partials + (size_t)item * G * kPartStride);
    }
    __syncthreads();
    if (trace && tid == 0) trace[4] = globaltimer();
    grid_barrier(p, S);  // every chunk partial is written
    if (trace && tid == 0) trace[5] = globaltimer();
    reduce_phase(p, S);
    if (trace && tid == 0) trace[6] = globaltimer();
  }
};

template <typename T, int G, bool PAGED>
__global__ void __launch_bounds__(kThreads, 1) step_kernel(const __grid_constant__ StepParams p) {
  Step<T, G, PAGED>::run(p);
}

}  // namespace mac
