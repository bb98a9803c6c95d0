// mac_step.cuh -- the span kernel: one persistent kernel per decode step
// (cooperative launch, one CTA per SM) for GQA groups of up to four query
// heads (groups of eight run the ring kernel, mac_ring.cuh): eight consumer
// warps and one producer warp.
//
//   Phase M (Match, [MAC] "Match (2)"/"Match (3)", K1): the pre-RoPE query
//   rings of all (request, head) pairs form B*Hq*K rows, cut into chunks of at
//   most a stage (never across heads) dealt round-robin to the CTAs, so every
//   CTA reads every part of the memory.  Eight lanes share a row; each sums
//   (a-b)^2 of its 16 elements in a pairwise tree (a-b of two bf16 values is
//   exact in fp32) and the eight finish the tree with shuffles, so a distance
//   carries at most 8 roundings of non-negative terms.  The pages' expansion
//   |a|^2+|b|^2-2a.b cancels badly for close pairs and is not used.  Each warp
//   combines its rows' best (distance, position) into the head's minimum with
//   a 64-bit atomic max of a packed key, a total order (smaller distance, then
//   more recent position), so the result does not depend on scheduling.
//
//   Complete (K2), tail pieces: the last r tokens of every unit, which every
//   head attends whatever the match decides, so they run before the
//   decisions exist (their tiles are copied during the match).
//
//   Grid barrier; every CTA turns the minima into decisions ([MAC] K1: hit
//   iff the smallest squared distance is strictly below thr^2) and lays out
//   the band [s, m-r] of every unit (request, kv head), s = the first token
//   any head of the unit needs (p-r+1 for a hit at p, 1 for a miss).  Band
//   pieces follow; a head whose band starts after s masks the tokens before
//   its own start ([MAC] "GQA intra-group skew").
//
//   Merge: the CTA that finishes a unit's last piece (a count per unit)
//   merges, per head, the cached rectified summary of a hit, the band
//   pieces in token order (giving AS_{1:m-r}) and then the tail pieces
//   (giving the output); a unit without band pieces is merged after the
//   decisions by one CTA chosen by its index.
//
// Work balance ("span-balanced" flash decode): the tail tokens of all units
// are laid end to end and cut into one contiguous span per CTA, and so are
// the band tokens; a span meets a few units, and each meeting (a piece)
// leaves one partial summary (running max, sum, weighted values; base-2 log
// domain, [MAC] "Complete").  A GQA group loads each K/V tile once for its G
// query heads.  Full attention (and ring seeding) run the same pieces with
// s = 1 and no match, so a decode step whose heads all miss is bitwise equal
// to full attention.
//
// Streaming: one ring of kStages shared-memory stages filled with 1-D TMA
// bulk copies by the producer warp (full/empty mbarriers) and drained by the
// consumer warps.  Every wait is bounded and reports MAC_DEV_WAIT_TIMEOUT
// instead of hanging.
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

__device__ __forceinline__ unsigned long long atom_add_release_u64(unsigned long long *p, unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.add.release.gpu.global.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
  return old;
}

// A count of finished pieces: release of the partials the calling CTA wrote
// before its consumer barrier, acquire of those the earlier counts released.
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

// SINK: whether the kernel attends front-sink pieces (a launch with a front
// sink uses the SINK = true kernels; the others carry none of that code).
// TRACE: whether it records the phase trace (mac_set_trace); the product
// kernels carry none of that code either.
template <typename T, int G, bool PAGED, bool SINK, bool TRACE = false>
struct Step {
  static constexpr int kRowBytes = kHeadDim * (int)sizeof(T);
  static constexpr int kTileTok = kStageBytes / (2 * kRowBytes);  // 64 (bf16) / 32 (fp32)
  static constexpr int kMatchRows = kStageBytes / kRowBytes;      // ring rows per stage
  static constexpr int kRPG = kMatchRows / 32;                    // rows per lane group per match chunk
  static constexpr int kLogRPG = ilog2c(kRPG);
  static constexpr int kPer = 16 / (int)sizeof(T);                // elements per 16-byte piece
  static constexpr int kNP = 16 / kPer;                           // pieces per lane (16 dims)
  static constexpr int kPairs = 8;                                // float2 pairs per lane (16 dims)
  // attention: a half-warp (16 lanes, 8 dims each) per token; kAGroups
  // half-warps per CTA, kATPG tokens each per tile
  static constexpr int kAGroups = kWarps * 2;
  static constexpr int kATPG = kTileTok / kAGroups;               // 4 (bf16) / 2 (fp32)
  static constexpr int kAPairs = 4;                               // float2 pairs per lane (8 dims)
  static constexpr int kALoads = 8 * (int)sizeof(T) / 16;         // 16-byte loads per lane and row
  static constexpr int kAV = kATPG * G;                           // scores of a half-warp per tile
  static constexpr int kAScat = ilog2c(kAV);                      // reduce-scatter levels
  static constexpr int kAPlain = 4 - kAScat;                      // plain butterfly levels after them
  static constexpr int kLogG = ilog2c(G);
  static constexpr int kLogATPG = ilog2c(kATPG);
  static constexpr int kQBytes = G * kRowBytes;
  // per-stage side buffer: a tile's G query rows, or a match chunk's query
  // row, ring positions and chunk coordinates (int4 at kInfoOff)
  static constexpr int kInfoOff = kRowBytes + 4 * kMatchRows;
  static constexpr int kAux = (kQBytes > kInfoOff + 16 ? kQBytes : kInfoOff + 16);
  static constexpr int kOutPer = (G * kHeadDim + kConsumers - 1) / kConsumers;
  static_assert(kAV <= 16 && kAV >= 2, "one score per lane of a half-warp at most");

  // dynamic shared memory layout
  static constexpr size_t kOffQ = (size_t)kStages * kStageBytes;
  static constexpr size_t kOffBar = kOffQ + (size_t)kStages * kAux;       // full[kStages], empty[kStages]
  static constexpr size_t kOffQrot = kOffBar + 128;                        // [G][d] f32
  static constexpr size_t kOffRedO = kOffQrot + 4 * (size_t)G * kHeadDim;  // [kWarps][4][G][d]
  static constexpr size_t kOffRedL = kOffRedO + 4 * (size_t)kWarps * 4 * G * kHeadDim;
  static constexpr size_t kOffRedM = kOffRedL + 4 * (size_t)kWarps * 4 * G;
  static constexpr size_t kOffX = kOffRedM + 4 * (size_t)kWarps * G;
  static_assert(kOffBar % 8 == 0 && kOffX % 8 == 0, "alignment");

  // X: the matched position of every head (-1: miss)
  __host__ __device__ static int x_ints(int B, int Hq, int K) { (void)K; return B * Hq; }
  __host__ __device__ static size_t off_units(int B, int Hq, int K) {
    return (kOffX + 4 * (size_t)x_ints(B, Hq, K) + 7) / 8 * 8;
  }
  // + offsets of the tail and long-band segments and the short-band cost
  // prefix (int64, n_units + 1 each), query position, band start and the
  // short-band list (int32) and the tail and band CTA runs (short2) of every
  // unit, then the RoPE cos/sin table of every request when there are at
  // most kRopeTab of them
  __host__ __device__ static size_t off_rope(int B, int Hq, int Hkv, int K) {
    const size_t U = (size_t)B * Hkv;
    return (off_units(B, Hq, K) + 24 * (U + 1) + 20 * U + 7) / 8 * 8;
  }
  __host__ __device__ static size_t smem_bytes(int B, int Hq, int Hkv, int K) {
    const size_t tab = B <= kRopeTab ? 8 * (size_t)B * (kHeadDim / 2) : 0;
    return off_rope(B, Hq, Hkv, K) + tab;
  }

  struct Smem {
    uint8_t *stage;     // [kStages][kStageBytes]
    uint8_t *qbuf;      // [kStages][kAux]: pre-RoPE query rows of a piece's unit, or a
                        // match chunk's query row and ring positions
    uint64_t *full;     // [kStages]: the stage's copy has landed
    uint64_t *empty;    // [kStages]: every consumer warp is done with the stage
    float *qrot;        // [G][d]: rotated, scaled query of the current piece
    float *red_o;       // [kWarps][4][G][d]
    float *red_l;       // [kWarps * 4][G]
    float *red_m;       // [kWarps][G]
    int32_t *X;
    int64_t *offA;      // [n_units + 1]: first global index of each unit's tail segment
    int64_t *offB;      // [n_units + 1]: same for the long bands on their cost axis: each
                        // long band is kLongPiece (a piece's fixed cost) + its tokens;
                        // short ones count 0
    int64_t *spanA;     // [grid + 1]: CTA c's tail span is [spanA[c], spanA[c+1])
    int64_t *spanB;     // [grid + 1]: same for the long bands
    int *neA, *neB;     // [grid + 1]: non-empty spans among CTAs 0..c-1
    int32_t *u_pos;     // [n_units]: position of the unit's query (RoPE angle pos - 1)
    int32_t *u_s;       // [n_units]: first band token of the unit
    int32_t *shortU;    // [n_units]: the units with a short band, in unit order
    int64_t *scp;       // [n_units + 1]: prefix of their costs (tokens + kPieceCost)
    short2 *runA;       // [n_units]: first and last CTA meeting the unit's tail (x > y: none)
    short2 *runB;       // [n_units]: same for its long band
    int *n_short;       // their number; CTA c has entries [c*n/P, (c+1)*n/P)
    long long *scan;    // [kWarps]: block_scan's warp totals
    long long *short_max;  // longest band that is one piece
    long long *band_tot;   // [2]: long-band tokens, their cost plus the short pieces'
    float2 *rope;       // [B][d/2]: cos, sin of the query's rotation angles (B <= kRopeTab), or null
    int *mask;          // [kStages]: valid 16-row groups of the tile in the stage (pages, if paged)
    volatile int *abort;
    volatile int *ready;  // layouts known to the producer: 1 tails (and bands in full mode), 2 bands
    volatile uint32_t *issued;  // uses the producer copied (published at its end)
    int rpar;                   // decode: the copy of the ring's match state in use
    volatile int *last;         // this CTA finished the last piece of a unit
  };

  struct Piece {
    int u, lo, hi;
    int sink;  // the front sink [1, min(F, m)] of unit u (an output-only piece)
  };

  // Phase trace point (see mac_set_trace): thread 0 records %globaltimer.
  // Like every region run by one thread, it ends with the warp reconverged
  // before the barriers and shuffles that follow.
  __device__ static void stamp(unsigned long long *trace, int k) {
    if constexpr (TRACE) {
      if (trace && threadIdx.x == 0) trace[k] = globaltimer();
      __syncwarp();
    }
  }
  __device__ static unsigned long long *cta_trace(const StepParams &p) {
    if constexpr (TRACE) return p.trace ? p.trace + (size_t)blockIdx.x * kTracePoints : nullptr;
    return nullptr;
  }

  // Lane `sub` (0..7) of a token's 8-lane group owns 16 dimensions: piece c
  // covers dims [c*8*kPer + sub*kPer, +kPer), so each group reads 128
  // contiguous bytes of a row per piece (no shared-memory bank conflicts).
  __device__ static int piece_dim(int c, int sub) { return c * 8 * kPer + sub * kPer; }

  // the lengths the scratch and the cache hold
  __device__ static bool len_ok(const StepParams &p, int64_t m) { return m >= 1 && m <= p.max_len; }
  __device__ static int64_t unit_len(const StepParams &p, const Smem &S, int u) {
    return (int64_t)S.u_pos[u] - p.len_sub;
  }

  // ---------------------------------------------------------------------
  // segments, spans and pieces
  // ---------------------------------------------------------------------

  // First token of unit u's segment: tails [max(F+1, m-r+1), m], bands
  // [s, m-r] (F: the front sink, 0 without one).
  __device__ static int64_t seg_first(const StepParams &p, const Smem &S, int ph, int u) {
    if (ph == 1) return S.u_s[u];
    const int64_t a = unit_len(p, S, u) - p.r + 1;
    return a > p.sink_f + 1 ? a : p.sink_f + 1;
  }
  __device__ static int64_t seg_len(const StepParams &p, const Smem &S, int ph, int u) {
    const int64_t m = unit_len(p, S, u);
    if (!len_ok(p, m)) return 0;
    if (ph == 0) {
      const int64_t n = m - seg_first(p, S, 0, u) + 1;
      return n > 0 ? n : 0;
    }
    const int64_t n = (m - p.r) - (int64_t)S.u_s[u] + 1;
    return n > 0 ? n : 0;
  }

  __device__ static const int64_t *offs(const Smem &S, int ph) { return ph ? S.offB : S.offA; }

  // c * total / P, in 32-bit arithmetic whenever the product fits (the
  // common case: 64-bit division is a long serial routine)
  __device__ static int64_t part_of(int c, int64_t total, int P) {
    if (total < (1LL << 23)) return (int64_t)((uint32_t)c * (uint32_t)total / (uint32_t)P);
    return div_s64((int64_t)c * total, P);
  }
  __device__ static const int64_t *spans(const Smem &S, int ph) { return ph ? S.spanB : S.spanA; }

  // the CTA whose (non-empty) span holds global index x (x < total): the
  // last c < P with span[c] <= x (span[0] = 0), by binary lifting over the
  // P <= kMaxGrid entries: a fixed number of steps without branches
  __device__ static int cta_of(const int64_t *span, int P, int64_t x) {
    int lo = 0;
#pragma unroll
    for (int s = kMaxGrid / 2; s >= 1; s >>= 1) {
      const int t = lo + s;
      if (t < P && span[t] <= x) lo = t;
    }
    return lo;
  }
  // unit whose segment holds global index g (g < T): the last u < U with
  // off[u] <= g, by binary lifting
  __device__ static int unit_of(const int64_t *off, int U, int64_t g) {
    int lo = 0;
#pragma unroll 1
    for (int s = U > 1 ? 1 << (31 - __clz(U - 1)) : 0; s >= 1; s >>= 1) {
      const int t = lo + s;
      if (t < U && off[t] <= g) lo = t;
    }
    return lo;
  }

  // The first piece of span [g0, g1) at unit >= u; false when none is left.
  __device__ static bool find_piece(const StepParams &p, const Smem &S, int ph, int u, int64_t g0,
                                    int64_t g1, Piece *pc) {
    const int64_t *off = offs(S, ph);
    const int U = p.B * p.Hkv;
#pragma unroll 1
    for (; u < U; ++u) {
      const int64_t a0 = off[u], z0 = off[u + 1];
      if (a0 >= g1) return false;
      const int64_t r0 = ph && z0 > a0 ? a0 + kLongPiece : a0;  // the band's first real token
      const int64_t a = r0 > g0 ? r0 : g0, z = z0 < g1 ? z0 : g1;
      if (a < z) {
        const int64_t t0 = seg_first(p, S, ph, u);
        pc->u = u;
        pc->lo = (int)(t0 + (a - r0));
        pc->hi = (int)(t0 + (z - r0) - 1);
        return true;
      }
    }
    return false;
  }

  // Tail layout, by all consumer threads (ends with a consumer barrier): the
  // exclusive prefix of the tail lengths, the CTA spans, their non-empty
  // counts and every unit's CTA run.  With at most as many units as CTAs,
  // unit u owns the CTAs [u*P/U, (u+1)*P/U) and its tail is cut evenly among
  // the first k' of them, k' = min(its CTAs, length / kMinTail rounded up),
  // so no CTA meets two units (a second piece would double its fixed costs)
  // nor gets a sliver, and everything but the prefix has a closed form; with
  // more units the tails, laid end to end, are cut into equal spans.
  static constexpr int kMinTail = 64;  // tokens: a tail piece worth its fixed cost
  static constexpr int kMinSpan = 64;  // tokens: a long-band span worth its fixed cost
  __device__ static int tail_ctas(int64_t len, int k) {
    if (len <= 0) return 0;
    const int64_t want = (len + kMinTail - 1) / kMinTail;
    return want < k ? (int)want : k;
  }
  __device__ static void layout_tails(const StepParams &p, const Smem &S) {
    int64_t *off = S.offA;
    const int U = p.B * p.Hkv, tid = threadIdx.x, P = gridDim.x;
    const bool aligned = U <= P;
    // prefix of (length << 9 | non-empty spans of the unit's CTAs); a
    // unit's k' <= P <= 256 used CTAs all hold non-empty spans
    long long carry = 0;
#pragma unroll 1
    for (int base = 0; base < U; base += kConsumers) {
      const int u = base + tid;
      long long x = 0;
      if (u < U) {
        const long long len = seg_len(p, S, 0, u);
        const int k = aligned ? (u + 1) * P / U - u * P / U : 0;
        x = (len << 9) | (long long)tail_ctas(len, k);
      }
      long long tot;
      const long long ex = block_scan(S, x, &tot);
      if (u < U) {
        off[u + 1] = (carry + ex + x) >> 9;
        if (aligned) S.neA[u + 1] = (int)((carry + ex + x) & 511);  // per-unit prefix, per-CTA below
      }
      carry += tot;
    }
    const int64_t total = carry >> 9;
    if (tid == 0) {
      off[0] = 0;
      if (aligned) S.neA[0] = 0;
    }
    consumer_sync();
    const int c = tid;  // P <= kMaxGrid = kConsumers: one CTA per thread (CTA P by thread 0)
    if (aligned) {
      int ne = 0;
      if (c < P) {
        const int u = ((c + 1) * U - 1) / P;
        const int a = u * P / U, j = c - a;
        const int64_t len = off[u + 1] - off[u];
        const int k = tail_ctas(len, (u + 1) * P / U - a);
        int64_t share = len;  // CTAs past the k' used ones: empty spans at the unit's end
        if (j < k)
          share = len < (1LL << 22) ? (int64_t)((uint32_t)len * (uint32_t)j / (uint32_t)k) : div_s64(len * j, k);
        S.spanA[c] = off[u] + share;
        // slices 0..j-1 of the unit: all non-empty up to the k' used ones
        ne = S.neA[u] + (j < k ? j : k);
      }
      const int neP = (int)(carry & 511);
      consumer_sync();  // every per-unit prefix read before the per-CTA counts overwrite it
      if (c < P) S.neA[c] = ne;
      if (c == 0) {
        S.spanA[P] = total;
        S.neA[P] = neP;
      }
#pragma unroll 1
      for (int u = tid; u < U; u += kConsumers) {
        const int a = u * P / U, k = tail_ctas(off[u + 1] - off[u], (u + 1) * P / U - a);
        S.runA[u] = k > 0 ? make_short2((short)a, (short)(a + k - 1)) : make_short2(0, -1);
      }
    } else {
      if (c <= P) S.spanA[c] = c < P ? part_of(c, total, P) : total;
      consumer_sync();
      int tot;
      const int ef = flag_scan(S, c < P && S.spanA[c] < S.spanA[c + 1], &tot);
      if (c < P) S.neA[c] = ef;
      if (c == 0) S.neA[P] = tot;
#pragma unroll 1
      for (int u = tid; u < U; u += kConsumers) S.runA[u] = find_run(S, 0, u);
    }
    consumer_sync();
  }

  // Band layout.  A band of at most max(kShortBand, all band tokens / P)
  // tokens (a hit whose match is recent: the common case) is one piece on
  // its own, since splitting it would cost more merges than it saves -- as
  // long as at most P/2 units qualify, else the bound is kShortBand (many
  // whole units dealt by count would give some CTAs two where spans give
  // each its exact share).  These short bands are dealt out in unit order,
  // CTA c taking list entries [c*n/P, (c+1)*n/P).  The long bands (misses,
  // old matches) are laid end to end and cut into CTA spans: the token
  // count of all bands plus kPieceCost per short piece is split evenly over
  // the CTAs, and each CTA's span is its share less its short pieces' cost.
  // So neither a run of short bands nor a long band piles up on a CTA.
  //
  // Two parts, each by one warp: band_units_warp (band starts, the short
  // list, long-band offsets) right after the decisions, so that the short
  // pieces can start; band_spans_block (the long-band spans, their
  // non-empty counts and every long unit's CTA run) by all consumer threads
  // while the producer copies the short pieces.  kShortBand, kPieceCost and
  // kLongPiece were set by timing the 4 x 128K decode step over a sweep of
  // each (the other two in their ranges made it no faster).
  static constexpr int kShortBand = 256;
  static constexpr int kPieceCost = 512;  // fixed cost of a piece and its merge, in tokens
  static constexpr int kSnap = 192;       // largest move of a long-band CTA boundary, in tokens
  // On the long bands' cost axis each band starts with kLongPiece virtual
  // tokens, a piece's fixed cost: a CTA whose span meets a band's start
  // pays it, so a CTA with two pieces gets fewer tokens.  No CTA boundary
  // falls inside that prefix or at its end (it moves to the band's start),
  // so every non-empty span holds real tokens of each band it meets.
  static constexpr int kLongPiece = 256;
  __device__ static bool short_band(const StepParams &p, const Smem &S, int u) {
    const int64_t n = seg_len(p, S, 1, u);
    return n > 0 && n <= *S.short_max;
  }
  __device__ static void short_range(const Smem &S, int *j0, int *j1) {
    const int ns = *S.n_short, c = blockIdx.x, P = gridDim.x;
    *j0 = c * ns / P;
    *j1 = (c + 1) * ns / P;
  }
  __device__ static Piece short_piece(const StepParams &p, const Smem &S, int j) {
    Piece pc;
    pc.sink = 0;
    pc.u = S.shortU[j];
    pc.lo = S.u_s[pc.u];
    pc.hi = (int)(unit_len(p, S, pc.u) - p.r);
    return pc;
  }
  __device__ static void band_units_warp(const StepParams &p, const Smem &S) {
    const int U = p.B * p.Hkv, lane = threadIdx.x & 31, P = gridDim.x;
    const bool decode = p.mode == MODE_DECODE;
    // each unit's band start and length (a 32-bit count: m < 2^31), the
    // length parked in shortU until the list overwrites it (entry j <= u,
    // written after every lane of the chunk has read its own)
    long long all = 0;
#pragma unroll 1
    for (int base = 0; base < U; base += 32) {
      const int u = base + lane;
      int len = 0;
      if (u < U) {
        if (decode) {
          int st = 0x7fffffff;
#pragma unroll
          for (int hh = 0; hh < G; ++hh) {
            const int pp = S.X[u * G + hh];  // head b*Hq + g*G + hh of unit u = b*Hkv + g
            st = min(st, pp >= 1 ? max(pp - p.r + 1, p.sink_f + 1) : p.sink_f + 1);
          }
          S.u_s[u] = st;
        }
        len = (int)seg_len(p, S, 1, u);
        S.shortU[u] = len;
      }
      // the chunk's sum from two 16-bit halves (no 32-bit overflow)
      all += ((long long)__reduce_add_sync(kFull, (unsigned)len >> 16) << 16) +
             __reduce_add_sync(kFull, (unsigned)len & 0xffffu);
    }
    int smax = kShortBand;  // max(all / P, kShortBand)
    if (all >= (long long)(kShortBand + 1) * P) {
      const long long q = all < 0x7fffffffLL ? (long long)((unsigned)all / (unsigned)P) : div_s64(all, P);
      smax = q < 0x7fffffffLL ? (int)q : 0x7fffffff;
    }
    if (smax > kShortBand) {
      int cnt = 0;
#pragma unroll 1
      for (int base = 0; base < U; base += 32) {
        const int u = base + lane;
        const int len = u < U ? S.shortU[u] : 0;
        cnt += __popc(__ballot_sync(kFull, len > 0 && len <= smax));
      }
      if (cnt > P / 2) smax = kShortBand;
    }
    long long cb = 0, cc = 0;  // carries: long tokens, short costs
    int ns = 0;
#pragma unroll 1
    for (int base = 0; base < U; base += 32) {
      const int u = base + lane;
      const int len = u < U ? S.shortU[u] : 0;
      const bool sh = len > 0 && len <= smax;
      long long x = sh || len == 0 ? 0 : kLongPiece + len, y = sh ? len + kPieceCost : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long x2 = __shfl_up_sync(kFull, x, o), y2 = __shfl_up_sync(kFull, y, o);
        if (lane >= o) {
          x += x2;
          y += y2;
        }
      }
      const unsigned bal = __ballot_sync(kFull, sh);
      if (u < U) {
        S.offB[u + 1] = cb + x;
        S.runB[u] = make_short2(0, -1);  // no CTA run (band_runs_block marks the long bands')
      }
      if (sh) {
        const int j = ns + __popc(bal & ((1u << lane) - 1u));
        S.shortU[j] = u;
        S.scp[j + 1] = cc + y;
      }
      cb += __shfl_sync(kFull, x, 31);
      cc += __shfl_sync(kFull, y, 31);
      ns += __popc(bal);
    }
    if (lane == 0) {
      S.offB[0] = 0;
      S.scp[0] = 0;
      *S.n_short = ns;
      *S.short_max = smax;
      S.band_tot[0] = cb;       // long-band cost (tokens + a piece's cost per band)
      S.band_tot[1] = cb + cc;  // all cost
    }
    __syncwarp();
  }

  // Exclusive prefix count of one flag per consumer thread, in thread
  // order, and the total (both to every thread), from the warps' ballots.
  // It holds one consumer barrier; the caller's next consumer barrier must
  // come before the next use of the warp totals.
  __device__ static int flag_scan(const Smem &S, bool f, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned bal = __ballot_sync(kFull, f);
    if (lane == 0) S.scan[warp] = __popc(bal);
    consumer_sync();
    int base = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const int v = (int)S.scan[w];
      base += w < warp ? v : 0;
      tot += v;
    }
    *total = tot;
    return base + __popc(bal & ((1u << lane) - 1u));
  }

  // Exclusive scan of one value per consumer thread, in thread order, and
  // the total (both returned to every thread).  All consumer threads call
  // it; it holds two consumer barriers.
  __device__ static long long block_scan(const Smem &S, long long x, long long *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    long long xi = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(kFull, xi, o);
      if (lane >= o) xi += y;
    }
    if (lane == 31) S.scan[warp] = xi;
    consumer_sync();
    long long base = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const long long v = S.scan[w];
      base += w < warp ? v : 0;
      tot += v;
    }
    consumer_sync();
    *total = tot;
    return base + xi - x;
  }

  // The long-band spans (CTA c = consumer thread c), by all consumer threads
  // (ends with a consumer barrier).
  __device__ static void band_spans_block(const StepParams &p, const Smem &S) {
    const int c = threadIdx.x, P = gridDim.x;
    const int ns = *S.n_short;
    const long long tb = S.band_tot[0], tv = S.band_tot[1];
    // the long bands use the first Pl CTAs, each with at least kMinSpan
    // tokens of the cost axis (slivers cost a whole piece and a bigger merge)
    const long long want = (tv + kMinSpan - 1) / kMinSpan;
    const int Pl = want < P ? (int)(want > 0 ? want : 1) : P;
    long long cap = 0, tot;
    if (c < Pl) {
      const int j0 = c * ns / P, j1 = (c + 1) * ns / P;
      cap = part_of(c + 1, tv, Pl) - part_of(c, tv, Pl) - (S.scp[j1] - S.scp[j0]);
      cap = cap > 0 ? cap : 0;
    }
    long long st = block_scan(S, cap, &tot);
    st = st < tb ? st : tb;
    // a CTA boundary within kSnap tokens (and half a share) of a long
    // unit's boundary moves onto it: the CTAs on either side then hold one
    // piece each instead of one of them two, a piece's fixed cost being
    // worth more than the imbalance.  Moving every boundary to its nearest
    // unit boundary, when near enough, keeps the boundaries in order.
    if (c > 0 && c < P && st > 0 && st < tb) {
      const long long share2 = part_of(1, tv, 2 * Pl), half = share2 < kSnap ? share2 : kSnap;
      const int u = unit_of(S.offB, p.B * p.Hkv, st);
      const long long lo = S.offB[u], hi = S.offB[u + 1];
      if (st - lo <= kLongPiece) {
        st = lo;  // inside or at the end of the band's cost prefix
      } else if (st - lo <= hi - st) {
        if (st - lo <= half) st = lo;
      } else if (hi - st <= half) {
        st = hi;
      }
    }
    if (c < P) S.spanB[c] = st;
    if (c == 0) S.spanB[P] = tb;
    consumer_sync();
  }

  // The long-band spans' non-empty counts and every long unit's CTA run, by
  // all consumer threads (ends with a consumer barrier): only the merges
  // read them, so they are made while the first band tiles are in flight.
  __device__ static void band_runs_block(const StepParams &p, const Smem &S) {
    const int U = p.B * p.Hkv, c = threadIdx.x, P = gridDim.x;
    int tot;
    const int ef = flag_scan(S, c < P && S.spanB[c] < S.spanB[c + 1], &tot);
    if (c < P) S.neB[c] = ef;
    if (c == 0) S.neB[P] = tot;
    // Every long band's run, scattered from the non-empty spans: span c
    // holds global index x iff span[c] <= x < span[c+1] (the CTA cta_of
    // finds), so CTA c's thread marks the bands whose segment starts or ends
    // in its span -- each start and each end lies in exactly one.  One
    // search over the units per thread replaces two over the CTAs per band.
    if (c < P && S.spanB[c] < S.spanB[c + 1]) {
      const int64_t a = S.spanB[c], z = S.spanB[c + 1], *off = S.offB;
#pragma unroll 1
      for (int u = unit_of(off, U, a); u < U && off[u] < z; ++u) {
        if (off[u + 1] <= off[u]) continue;  // no long band
        if (off[u] >= a) S.runB[u].x = (short)c;
        if (off[u + 1] - 1 < z) S.runB[u].y = (short)c;
      }
    }
    consumer_sync();
  }

  // ---------------------------------------------------------------------
  // producer
  // ---------------------------------------------------------------------

  // The G pre-RoPE query rows of unit u's heads into stage st's side buffer.
  __device__ static void copy_q(const StepParams &p, const Smem &S, int st, int u, uint32_t bar) {
    const uint8_t *q = (const uint8_t *)p.q;
    const int b = u / p.Hkv, g = u % p.Hkv;
    const int64_t bh0 = (int64_t)b * p.Hq + g * G;
    if (p.q_stride == kHeadDim && p.q_offset == 0) {  // the group's G rows are contiguous
      bulk_g2s(smem_addr(S.qbuf + (size_t)st * kAux), q + (size_t)bh0 * kRowBytes, kQBytes, bar);
    } else {
      for (int hh = 0; hh < G; ++hh)
        bulk_g2s(smem_addr(S.qbuf + (size_t)st * kAux + hh * kRowBytes),
                 q + (size_t)((bh0 + hh) * p.q_stride + p.q_offset) * sizeof(T), kRowBytes, bar);
    }
  }

  // Paged tile of piece pc starting after token tb (a page boundary), with
  // the ids of its kSlots page-table slots from tb / 16 on already loaded
  // (kNoPage past the table): the rows of each 16-token page that fall in
  // the piece, page by page; an id outside the pool is refused and reported.
  static constexpr int32_t kNoPage = (int32_t)0x80000000;
  static constexpr int kSlots = kTileTok / 16;  // pages in a tile
  __device__ static void issue_paged_tile(const StepParams &p, const Smem &S, int st, const Piece &pc, int tb,
                                          bool with_q, const int32_t *ids) {
    const int g = pc.u % p.Hkv;
    uint8_t *kbuf = S.stage + (size_t)st * kStageBytes;
    const uint32_t bar = smem_addr(&S.full[st]);
    uint32_t bytes = with_q ? (uint32_t)kQBytes : 0u;
    int msk = 0;
#pragma unroll
    for (int pg = 0; pg < kSlots; ++pg) {
      const int pa = tb + pg * 16 + 1, ra = pa > pc.lo ? pa : pc.lo, rz = pa + 15 < pc.hi ? pa + 15 : pc.hi;
      if (ra > rz || ids[pg] == kNoPage) continue;  // (past the table: nothing to copy)
      if (ids[pg] < 0 || ids[pg] >= p.kv.n_pages) {
        set_status(p.ctl, MAC_DEV_BAD_PAGE);
        continue;
      }
      msk |= 1 << pg;
      bytes += 2u * (uint32_t)(rz - ra + 1) * kRowBytes;
    }
    S.mask[st] = msk;
    if (bytes == 0) {
      mbar_arrive(bar);
      return;
    }
    mbar_expect_tx(bar, bytes);
    if (with_q) copy_q(p, S, st, pc.u, bar);
    const unsigned long long pol = l2_evict_first_policy();
#pragma unroll
    for (int pg = 0; pg < kSlots; ++pg) {
      if (!((msk >> pg) & 1)) continue;
      const int pa = tb + pg * 16 + 1, ra = pa > pc.lo ? pa : pc.lo, rz = pa + 15 < pc.hi ? pa + 15 : pc.hi;
      const size_t off = (((size_t)ids[pg] * p.Hkv + g) * 16 + (size_t)(ra - pa)) * kRowBytes;
      const uint32_t nb = (uint32_t)(rz - ra + 1) * kRowBytes;
      uint8_t *dst = kbuf + (size_t)(ra - tb - 1) * kRowBytes;
      bulk_g2s_hint(smem_addr(dst), (const uint8_t *)p.kv.k + off, nb, bar, pol);
      bulk_g2s_hint(smem_addr(dst + kStageBytes / 2), (const uint8_t *)p.kv.v + off, nb, bar, pol);
    }
  }

  // Match chunk j: head j / cph, rows [(j % cph) * kMatchRows, +rows) of its
  // ring, cph = chunks per head (chunks never cross heads).
  __device__ static int chunks_per_head(int K) { return (K + kMatchRows - 1) / kMatchRows; }

  // Bounded spin of the producer lane on a shared flag set by a consumer.
  __device__ static bool wait_ready(const StepParams &p, const Smem &S, int level) {
    const long long t0 = clock64();
    while (*S.ready < level) {
      if (*S.abort) return false;
      if (clock64() - t0 > p.wait_limit) {
        set_status(p.ctl, MAC_DEV_WAIT_TIMEOUT);
        *S.abort = 1;
        return false;
      }
      __nanosleep(64);  // leave the issue slots to the warp doing the work
    }
    __threadfence_block();
    return true;
  }

  // Producer lane: wait for stage use n to be free, then arm its full barrier.
  // The run-out test's withheld use is never copied: the producer stalls
  // there (bounded) until the consumers' wait for it has run out.
  __device__ static bool acquire_stage(const StepParams &p, const Smem &S, uint32_t n) {
    if ((int)n == p.withhold) {
      const long long t0 = clock64();
      while (!*S.abort && clock64() - t0 <= 2 * p.wait_limit) {
      }
      if (!*S.abort) set_status(p.ctl, MAC_DEV_WAIT_TIMEOUT);
      *S.abort = 1;
      return false;
    }
    if (!mbar_wait_bounded(smem_addr(&S.empty[n % kStages]), ((n / kStages) & 1u) ^ 1u, S.abort, p.wait_limit)) {
      if (!*S.abort) set_status(p.ctl, MAC_DEV_WAIT_TIMEOUT);
      *S.abort = 1;
      return false;
    }
    return true;
  }

  // A piece's tiles, the same for the producer and the consumers: tile k
  // holds tokens tile_base + 1 .. tile_base + kTileTok.  In a contiguous
  // cache the first starts at the piece's first token, so a piece of
  // kTileTok tokens is one tile wherever it starts; in a paged cache it
  // starts with the page holding that token, so every tile is whole pages
  // (a page split between two tiles would cost a copy in each).
  __device__ static int tile_start(const Piece &pc) { return PAGED ? (pc.lo - 1) / 16 * 16 : pc.lo - 1; }
  __device__ static int tile_count(const Piece &pc) {
    return pc.hi >= pc.lo ? (pc.hi - 1 - tile_start(pc)) / kTileTok + 1 : 0;
  }
  __device__ static int tile_base(const Piece &pc, int k) { return tile_start(pc) + k * kTileTok; }

  // The tiles of one piece, from stage use n on; returns the next use.
  __device__ static uint32_t copy_piece(const StepParams &p, const Smem &S, const Piece &pc, uint32_t n) {
    const int nt = tile_count(pc);
    if (pc.u < 0 || pc.u >= p.B * p.Hkv || pc.lo < 1 || pc.hi < pc.lo || (!PAGED && pc.hi > p.kv.capacity)) {
      // a piece outside the cache is refused tile by tile: nothing is
      // copied and no row of its stages counts
#pragma unroll 1
      for (int k = 0; k < nt; ++k, ++n) {
        if (!acquire_stage(p, S, n)) break;
        set_status(p.ctl, MAC_DEV_BAD_COPY);
        S.mask[n % kStages] = 0;
        mbar_arrive(smem_addr(&S.full[n % kStages]));
      }
      return n;
    }
    if (PAGED) {
      // a table lookup per 16 rows: the next tile's page ids are loaded
      // (independent loads) before the wait for its stage
      const int32_t *row = p.kv.page_table + (int64_t)(pc.u / p.Hkv) * p.kv.max_pages;
      int32_t ids[kSlots], nxt[kSlots];
#pragma unroll
      for (int i = 0; i < kSlots; ++i) {
        const int64_t slot = (int64_t)(tile_base(pc, 0) / 16) + i;
        ids[i] = slot < p.kv.max_pages ? __ldg(row + slot) : kNoPage;
      }
#pragma unroll 1
      for (int k = 0; k < nt; ++k, ++n) {
#pragma unroll
        for (int i = 0; i < kSlots; ++i) {
          const int64_t slot = (int64_t)(tile_base(pc, k + 1) / 16) + i;
          nxt[i] = k + 1 < nt && slot < p.kv.max_pages ? __ldg(row + slot) : kNoPage;
        }
        if (!acquire_stage(p, S, n)) break;
        issue_paged_tile(p, S, n % kStages, pc, tile_base(pc, k), k == 0, ids);
#pragma unroll
        for (int i = 0; i < kSlots; ++i) ids[i] = nxt[i];
      }
      return n;
    }
    // contiguous cache, a piece inside it: checked once, then each tile is
    // two row ranges (the unit's K and V rows are contiguous)
    const size_t unit_off = (size_t)pc.u * (size_t)p.kv.capacity * kRowBytes;
    const uint8_t *kg = (const uint8_t *)p.kv.k + unit_off, *vg = (const uint8_t *)p.kv.v + unit_off;
    const unsigned long long pol = l2_evict_first_policy();
#pragma unroll 1
    for (int k = 0; k < nt; ++k, ++n) {
      if (!acquire_stage(p, S, n)) break;
      const int st = n % kStages;
      const int ra = tile_base(pc, k) + 1;  // the stage's first row
      const int rz = ra + kTileTok - 1 < pc.hi ? ra + kTileTok - 1 : pc.hi;
      const uint32_t nb = (uint32_t)(rz - ra + 1) * kRowBytes;
      const uint32_t bar = smem_addr(&S.full[st]);
      S.mask[st] = (1 << (kTileTok / 16)) - 1;  // (rows past pc.hi are excluded by position)
      mbar_expect_tx(bar, 2u * nb + (k == 0 ? (uint32_t)kQBytes : 0u));
      if (k == 0) copy_q(p, S, st, pc.u, bar);
      uint8_t *kbuf = S.stage + (size_t)st * kStageBytes;
      bulk_g2s_hint(smem_addr(kbuf), kg + (size_t)(ra - 1) * kRowBytes, nb, bar, pol);
      bulk_g2s_hint(smem_addr(kbuf + kStageBytes / 2), vg + (size_t)(ra - 1) * kRowBytes, nb, bar, pol);
    }
    return n;
  }

  // The ring's match state: the step count, the chunk counter and the
  // per-head minima of copy k (k = the step count's parity).
  __device__ static uint32_t *chunk_counter(const StepParams &p, int k) { return p.ring_ctl + 2 + k; }
  __device__ static unsigned long long *ring_best(const StepParams &p, int k) {
    return reinterpret_cast<unsigned long long *>(p.ring_ctl + 4) + (size_t)k * p.B * p.Hq;
  }

  // The match chunks this CTA takes from the ring's counter (chunk j: rows
  // [slot0, slot0 + rows) of head j / cph), each into the next stage use,
  // then one stage use with no rows that ends the match; returns the next
  // use.  CTAs that start earlier take more chunks.  The next chunk is taken
  // while the current one's stage is awaited.
  __device__ static uint32_t copy_match(const StepParams &p, const Smem &S, uint32_t n, int par) {
    const int cph = chunks_per_head(p.K), nc = p.B * p.Hq * cph;
    const unsigned long long pol = l2_evict_first_policy();
    uint32_t *ctr = chunk_counter(p, par);
    int j = (int)atomicAdd(ctr, 1u);
#pragma unroll 1
    for (;; ++n) {
      if (!acquire_stage(p, S, n)) return n;
      const int st = n % kStages;
      const uint32_t bar = smem_addr(&S.full[st]);
      uint8_t *side = S.qbuf + (size_t)st * kAux;
      if (j >= nc) {
        // the end of the match (plain store, ordered before the consumers'
        // wait by the arrive)
        *reinterpret_cast<int4 *>(side + kInfoOff) = make_int4(-1, 0, 0, 0);
        mbar_arrive(bar);
        return n + 1;
      }
      const int bh = j / cph, slot0 = (j % cph) * kMatchRows;
      const int rows = p.K - slot0 < kMatchRows ? p.K - slot0 : kMatchRows;
      const bool pos_copy = pos_by_copy(p);
      // the chunk's coordinates, then the head's query row and the chunk's
      // ring positions, into the side buffer
      *reinterpret_cast<int4 *>(side + kInfoOff) = make_int4(bh, slot0, rows, bh / p.Hq);
      mbar_expect_tx(bar, (uint32_t)rows * kRowBytes + kRowBytes + (pos_copy ? 4u * rows : 0u));
      bulk_g2s_hint(smem_addr(S.stage + (size_t)st * kStageBytes),
                    (const uint8_t *)p.ring_q + ((size_t)bh * p.K + slot0) * kRowBytes,
                    (uint32_t)rows * kRowBytes, bar, pol);
      bulk_g2s(smem_addr(side), (const uint8_t *)p.q + (size_t)((int64_t)bh * p.q_stride + p.q_offset) * sizeof(T),
               kRowBytes, bar);
      if (pos_copy)
        bulk_g2s(smem_addr(side + kRowBytes), p.ring_pos + (size_t)(bh / p.Hq) * p.K + slot0, 4u * rows, bar);
      j = (int)atomicAdd(ctr, 1u);
    }
  }
  // Ring positions come with the chunk when their rows are 16-byte aligned.
  __device__ static bool pos_by_copy(const StepParams &p) { return (p.K & 3) == 0; }

  // The producer warp: a copy engine.  Its first lane copies the match
  // chunks it takes from the ring's counter (they need nothing but the
  // parameters) and the use that ends the match, then the tail tiles once
  // the consumers publish the unit positions and the tail layout, the short
  // pieces once they publish the short-band list, and the long-band pieces
  // once they publish the long-band spans.  Every copy goes in the order the
  // consumers use the stages.
  __device__ static void producer_warp(const StepParams &p, const Smem &S) {
    const int lane = threadIdx.x & 31, U = p.B * p.Hkv;
    unsigned long long *tr = lane == 0 ? cta_trace(p) : nullptr;
    const bool decode = p.mode == MODE_DECODE;
    uint32_t n = 0;
    if (lane == 0) {
      if (decode) n = copy_match(p, S, 0, S.rpar);
      if (tr) tr[30] = globaltimer();
      if (!wait_ready(p, S, 1)) *S.abort = 1;  // unit positions and tail layout
      if (tr) tr[31] = globaltimer();
    }
    __syncwarp();
    if (decode && !PAGED) {
      // the tile a recent match's band needs (a hit at m-1 starts it at
      // m-r) into L2 while the match runs, for the units u = c mod P
#pragma unroll 1
      for (int u = blockIdx.x + lane * (int)gridDim.x; u < U; u += 32 * (int)gridDim.x) {
        const int64_t m = unit_len(p, S, u), hi = m - p.r;
        if (!len_ok(p, m) || hi < 1 || hi > p.kv.capacity) continue;
        const int64_t lo = hi - kTileTok + 1 > 1 ? hi - kTileTok + 1 : 1;
        const size_t off = ((size_t)u * (size_t)p.kv.capacity + (size_t)(lo - 1)) * kRowBytes;
        const uint32_t bytes = (uint32_t)(hi - lo + 1) * kRowBytes;
        bulk_prefetch_l2((const uint8_t *)p.kv.k + off, bytes);
        bulk_prefetch_l2((const uint8_t *)p.kv.v + off, bytes);
      }
    }
    if (lane == 0) {
      // tails (the unit layout is known), then the short bands and the long
      // bands as their layouts are published
#pragma unroll 1
      for (int kind = 0; kind < 3 && !*S.abort; ++kind) {
        if (kind == 1) {
          if (!wait_ready(p, S, 2)) break;
          if (tr) tr[26] = globaltimer();
        } else if (kind == 2) {
          if (tr) tr[9] = globaltimer();
          if (!wait_ready(p, S, 3)) break;
          if (tr) tr[27] = globaltimer();
        }
        PieceIter I = piece_iter(p, S, kind);
        Piece pc;
        while (!*S.abort && next_piece(p, S, I, pc)) n = copy_piece(p, S, pc, n);
      }
      __threadfence_block();
      *S.issued = n;
    }
    __syncwarp();
    if (decode && !*S.abort) copy_step_queries(p, S);
  }

  // The step's queries, rows bh = c + i P: into ring slot pos mod K (the
  // fused append; the final merge writes the slot's summary), or into the
  // ring workspace's staging area for the append kernel, so that the caller
  // may reuse its query buffer right away.  By the producer warp once its
  // copies are issued: the grid barrier (before the band layout it waited
  // for) ordered every match's ring reads before these writes.
  __device__ static void copy_step_queries(const StepParams &p, const Smem &S) {
    const int lane = threadIdx.x & 31;
    constexpr int kChunks = kHeadDim / kPer;  // 16-byte pieces of a row
#pragma unroll 1
    for (int bh = blockIdx.x; bh < p.B * p.Hq; bh += gridDim.x) {
      const int b = bh / p.Hq, u = b * p.Hkv + (bh - b * p.Hq) / G;
      const int pos = S.u_pos[u];
      const bool app = p.app_o && len_ok(p, pos);
      if (lane < kChunks && (app || !p.app_o)) {
        const uint4 qv = reinterpret_cast<const uint4 *>(p.q)[((int64_t)bh * p.q_stride + p.q_offset) / kPer + lane];
        if (app)
          reinterpret_cast<uint4 *>(p.app_q)[((int64_t)bh * p.K + pos % p.K) * kChunks + lane] = qv;
        else
          reinterpret_cast<uint4 *>(p.stage_q)[(int64_t)bh * kChunks + lane] = qv;
      }
    }
  }

  // Consumer side of stage use n.
  __device__ static bool wait_use(const StepParams &p, const Smem &S, uint32_t n) {
    const bool ok = mbar_wait_bounded(smem_addr(&S.full[n % kStages]), (n / kStages) & 1u, S.abort, p.wait_limit);
    if (!ok && !*S.abort) {
      set_status(p.ctl, MAC_DEV_WAIT_TIMEOUT);
      *S.abort = 1;
    }
    return ok;
  }
  __device__ static void release(const Smem &S, uint32_t n) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(smem_addr(&S.empty[n % kStages]));
  }

  // ---------------------------------------------------------------------
  // phase M
  // ---------------------------------------------------------------------

  // The lane's part of the squared L2 distance between the query and a row:
  // exact differences of its 16 elements (bf16), squares and a pairwise tree
  // (the 8 lanes of the group are summed by the caller).
  __device__ static float lane_dist(const uint8_t *row, int sub, const float2 *qv) {
    float2 df[kPairs];
#pragma unroll
    for (int c = 0; c < kNP; ++c) {
      const uint4 raw = *reinterpret_cast<const uint4 *>(row + c * 128 + sub * 16);
      if constexpr (sizeof(T) == 2) {
        // b - q straight from the bf16 element (one mixed-precision
        // subtraction each, exact widening then one rounding): the negation
        // of the difference, which squares to the same value
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 q = qv[c * 4 + k];
          df[c * 4 + k] = make_float2(bf16_minus_f32((uint16_t)(w[k] & 0xffffu), q.x),
                                      bf16_minus_f32((uint16_t)(w[k] >> 16), q.y));
        }
      } else {
        float2 e2[kPer / 2];
        unpack16x2<T>(raw, e2);
#pragma unroll
        for (int k = 0; k < kPer / 2; ++k) {
          const float2 q = qv[c * (kPer / 2) + k];
          df[c * (kPer / 2) + k] = __fadd2_rn(q, make_float2(-e2[k].x, -e2[k].y));
        }
      }
    }
    float2 t[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) t[k] = __ffma2_rn(df[k + 4], df[k + 4], __fmul2_rn(df[k], df[k]));
    t[0] = __fadd2_rn(t[0], t[2]);
    t[1] = __fadd2_rn(t[1], t[3]);
    t[0] = __fadd2_rn(t[0], t[1]);
    return __fadd_rn(t[0].x, t[0].y);
  }

  // The warp's best (distance, position) joins head bh's global minimum.
  // Scan the match chunk of stage use n: its rows, the head's query row, the
  // chunk's coordinates and (K a multiple of 4) the rows' positions all
  // arrive in the stage.  Each lane sums (a-b)^2 of its 16 elements of the
  // group's kRPG rows; a reduce-scatter over the group's 8 lanes (xor 4, 2,
  // then 1) leaves lanes 2k, 2k+1 with row k's distance (three pairwise
  // levels, as in row_dist); the warp's best then joins the head's minimum.
  // The match chunk in stage use n (false: the use that ends the match).
  // The warp's best candidate joins its head's minimum in the ring's copy.
  __device__ static bool match_chunk(const StepParams &p, const Smem &S, uint32_t n, int grp, int sub,
                                     unsigned long long &wait_ns, unsigned long long *best) {
    static_assert(kRPG == 4 || kRPG == 2, "rows per lane group");
    const bool pos_copy = pos_by_copy(p);
    const int kk = (sub >> (3 - kLogRPG)) & (kRPG - 1);  // the row this lane finishes
    const int i_mine = grp + 32 * kk;
    int pk_mine = 0;
    const bool timed = TRACE && threadIdx.x == 0 && p.trace;
    const unsigned long long tw = timed ? globaltimer() : 0ull;
    const bool ok = wait_use(p, S, n);
    if (timed) wait_ns += globaltimer() - tw;
    if (n == 0) stamp(cta_trace(p), 8);
    const int st = n % kStages;
    if (reinterpret_cast<const int4 *>(S.qbuf + (size_t)st * kAux + kInfoOff)->x < 0 || !ok) {
      release(S, n);  // the end of the match (or an aborted wait)
      return false;
    }
    const uint8_t *rows = S.stage + (size_t)st * kStageBytes;
    const uint8_t *side = S.qbuf + (size_t)st * kAux;
    const int4 info = *reinterpret_cast<const int4 *>(side + kInfoOff);  // bh, slot0, rows, b
    const int bh = info.x, cnt = info.z;
    float2 qv[kPairs];
#pragma unroll
    for (int cc = 0; cc < kNP; ++cc)
      unpack16x2<T>(*reinterpret_cast<const uint4 *>(side + cc * 128 + sub * 16), qv + cc * (kPer / 2));
    if (pos_copy)
      pk_mine = reinterpret_cast<const int32_t *>(side + kRowBytes)[i_mine < cnt ? i_mine : cnt - 1];
    else
      pk_mine = __ldg(p.ring_pos + (int64_t)info.w * p.K + info.y + (i_mine < cnt ? i_mine : cnt - 1));
    const int64_t m = S.X[info.w];  // the request's length, tabled before the match
    // the lane's partial sums of the group's rows (rows past the chunk read
    // stale stage bytes and are discarded below)
    float v[kRPG];
#pragma unroll
    for (int k = 0; k < kRPG; ++k) {
      const int i = grp + 32 * k;
      v[k] = lane_dist(rows + (size_t)(i < cnt ? i : cnt - 1) * kRowBytes, sub, qv);
    }
    // reduce-scatter: level xor 4 keeps half the rows, xor 2 (kRPG == 4)
    // the next half, xor 1 finishes the sum
#pragma unroll
    for (int lev = 0; lev < kLogRPG; ++lev) {
      const int off = 4 >> lev;
      const bool up = (threadIdx.x & off) != 0;
      const int half = kRPG >> (lev + 1);
#pragma unroll
      for (int i = 0; i < kRPG / 2; ++i) {
        if (i < half) {
          const float send = up ? v[i] : v[i + half];
          const float keep = up ? v[i + half] : v[i];
          v[i] = __fadd_rn(keep, __shfl_xor_sync(kFull, send, off));
        }
      }
    }
    float D = v[0];
#pragma unroll
    for (int lev = kLogRPG; lev < 3; ++lev) D = __fadd_rn(D, __shfl_xor_sync(kFull, D, 4 >> lev));
    int pos_lo = 1, pos_hi = 0;
    if (len_ok(p, m)) {
      pos_lo = m - p.K > 1 ? (int)(m - p.K) : 1;
      pos_hi = (int)(m - 1);
    }
    const bool valid = ok && i_mine < cnt && pk_mine >= pos_lo && pk_mine <= pos_hi;
    int bp = valid ? pk_mine : -1;
    D = valid ? D : INFINITY;
    release(S, n);
    // the warp's best: lanes 2k and 2k+1 agree, so xor 2 and up
#pragma unroll
    for (int off = 8 / kRPG; off <= 16; off <<= 1) {
      const float d2 = __shfl_xor_sync(kFull, D, off);
      const int p2 = __shfl_xor_sync(kFull, bp, off);
      if (better(d2, p2, D, bp)) {
        D = d2;
        bp = p2;
      }
    }
    if ((threadIdx.x & 31) == 0 && bp >= 1) atomicMax(&best[bh], pack_best(D, bp));
    return true;
  }

  // The match chunks the producer took for this CTA, from stage use n on,
  // up to and including the use that ends the match.  Nothing here touches
  // the scratch workspace, so it may run before the previous kernel on the
  // stream has finished.
  __device__ static void match_phase(const StepParams &p, const Smem &S, uint32_t &n) {
    const int ct = threadIdx.x, warp = ct >> 5, lane = ct & 31, sub = lane & 7;
    const int grp = warp * 4 + (lane >> 3);  // row group: rows grp, grp + 32, ... of a chunk
    unsigned long long *best = ring_best(p, S.rpar);
    unsigned long long wait_ns = 0;
    int chunks = 0;
#pragma unroll 1
    while (match_chunk(p, S, n++, grp, sub, wait_ns, best)) ++chunks;
    unsigned long long *tr = threadIdx.x == 0 ? cta_trace(p) : nullptr;
    if (tr) {
      tr[28] += wait_ns;
      tr[29] += (unsigned long long)chunks;
    }
  }

  // All CTAs of the (co-resident, cooperative) grid meet; bounded wait.  One
  // thread per CTA polls without sleeping: the last arrival is seen one L2
  // round trip after it lands.
  __device__ static void grid_barrier(const StepParams &p, const Smem &S) {
    // every consumer's earlier writes and atomics (the match minima, the
    // tail partials) come before thread 0's release
    consumer_sync();
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
    consumer_sync();
  }

  // Decisions of every head from the combined minima (one head per consumer
  // thread); the cached summaries of the hits are asked into L2 for the
  // merges; then, by warp 0, every unit's band start and the short-band list
  // (every CTA computes the same), after which the producer may copy short
  // pieces and lay out the long bands.  Ends with a consumer barrier.
  __device__ static void decide(const StepParams &p, const Smem &S, unsigned long long *trace) {
    const int tid = threadIdx.x, n_bh = p.B * p.Hq;
#pragma unroll 1
    for (int bh = tid; bh < n_bh; bh += kConsumers) {
      const int b = bh / p.Hq, u = b * p.Hkv + (bh % p.Hq) / G;
      const int64_t m = unit_len(p, S, u);
      const unsigned long long inv = __ldcg(&ring_best(p, S.rpar)[bh]);
      int pos = -1;
      if (inv != 0ull && len_ok(p, m) && m >= p.min_context) {
        const unsigned long long key = ~inv;
        const float d = __uint_as_float((uint32_t)(key >> 32));
        if (d < p.thr2) pos = (int)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
      }
      S.X[bh] = pos;
      if (blockIdx.x == 0 && p.match_pos_out) p.match_pos_out[bh] = pos;
      if (pos >= 1 && bh % gridDim.x == blockIdx.x) {
        const int64_t slot = (int64_t)bh * p.K + pos % p.K;
        for (int k = 0; k < kHeadDim * 4; k += 128)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(p.ring_o + slot * kHeadDim + k / 4));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p.ring_lse + slot));
      }
    }
    consumer_sync();
    stamp(trace, 5);
  }

  // Every unit's band start and the short-band list (warp 0), after which
  // the producer may copy short pieces, then the long-band spans (all
  // consumer threads), after which it may copy long-band pieces.  Ends with
  // a consumer barrier.
  __device__ static void layout_bands(const StepParams &p, const Smem &S, unsigned long long *trace) {
    if (threadIdx.x < 32) {
      band_units_warp(p, S);
      __threadfence_block();
      if (threadIdx.x == 0) *S.ready = 2;
      __syncwarp();
    }
    consumer_sync();
    band_spans_block(p, S);
    if (threadIdx.x == 0) {
      __threadfence_block();
      *S.ready = 3;
    }
    band_runs_block(p, S);
    (void)trace;
  }

  // ---------------------------------------------------------------------
  // attention over the CTA's pieces
  // ---------------------------------------------------------------------


  // cos, sin of rotation angle j of request b at position pos: from the
  // CTA's table when there is one, else computed here.
  __device__ static float2 rope_cs(const StepParams &p, const Smem &S, int b, int64_t pos, int j) {
    if (S.rope) return S.rope[b * (kHeadDim / 2) + j];
    float c, sn;
    rope_angle(pos, p.rope_f[j], &c, &sn);
    return make_float2(c, sn);
  }

  __device__ static void rotate_pair(float a, float b, float2 cs, float scale, float *ra, float *rb) {
    *ra = __fmul_rn(__fsub_rn(__fmul_rn(a, cs.x), __fmul_rn(b, cs.y)), scale);
    *rb = __fmul_rn(__fadd_rn(__fmul_rn(b, cs.x), __fmul_rn(a, cs.y)), scale);
  }

  // R(pos) q~ * log2(e)/sqrt(d) of the piece's G heads into shared memory,
  // from the pre-RoPE rows that came with its first tile: one rotation pair
  // per consumer thread (explicit roundings keep the result identical
  // wherever it is computed).  Ends with a consumer barrier.
  __device__ static void rotate_query(const StepParams &p, const Smem &S, int st, int b, int64_t pos) {
    const int half = kHeadDim / 2;
    const bool inter = p.rope_mode == MAC_ROPE_INTERLEAVED;
    for (int i = threadIdx.x; i < G * half; i += kConsumers) {
      const int hh = i / half, j = i % half;
      const int ia = inter ? 2 * j : j, ib = inter ? 2 * j + 1 : j + half;
      const void *row = S.qbuf + (size_t)st * kAux + hh * kRowBytes;
      const float a = elem_f32<T>(row, ia), bb = elem_f32<T>(row, ib);
      const float2 cs = p.rope_mode == MAC_ROPE_NONE ? make_float2(1.f, 0.f) : rope_cs(p, S, b, pos, j);
      float ra, rb;
      rotate_pair(a, bb, cs, p.q_scale, &ra, &rb);
      S.qrot[hh * kHeadDim + ia] = ra;
      S.qrot[hh * kHeadDim + ib] = rb;
      if (!(isfinite(a) && isfinite(bb))) set_status(p.ctl, MAC_DEV_NONFINITE_Q);
    }
    consumer_sync();
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

  // the lane's 8 dims (d = 8 sub .. 8 sub + 7) of row `row`
  __device__ static void row_dims(const uint8_t *base, int row, int sub, float2 (&f)[kAPairs]) {
#pragma unroll
    for (int c = 0; c < kALoads; ++c)
      unpack16x2<T>(*reinterpret_cast<const uint4 *>(base + row * kRowBytes + sub * 8 * (int)sizeof(T) + c * 16),
                    f + c * (kAPairs / kALoads));
  }

  // One piece: tokens [pc.lo, pc.hi] of unit pc.u for its G heads; the
  // piece's partial summary goes to dst ([G][kPartStride]).  A half-warp
  // takes one token of a kATPG-token slot of every tile; lane `sub` owns
  // dims 8 sub .. 8 sub + 7 of the rotated query (held in registers for the
  // whole piece) and of the weighted values.
  __device__ static void attend_piece(const StepParams &p, const Smem &S, uint32_t &n, int ph,
                                      const Piece &pc, float *dst, bool first_piece) {
    unsigned long long *trace = first_piece ? cta_trace(p) : nullptr;
    unsigned long long *tr_all = ph == 1 && threadIdx.x == 0 ? cta_trace(p) : nullptr;
    if (tr_all) {
      tr_all[22] += (unsigned long long)(pc.hi - pc.lo + 1);
      tr_all[23] += 1;
    }
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, sub = lane & 15;
    const int grp = warp * 2 + (lane >> 4);  // this half-warp: rows grp, grp + 16, ... of a tile
    const int idx = sub >> kAPlain;          // this lane's score slot
    const int ti = idx / G, hm = idx % G;    // its token (of the group's kATPG) and head
    const int b = pc.u / p.Hkv, g = pc.u % p.Hkv;
    int lo_mine = pc.lo;                     // first token of the lane's head in this piece
    if (ph == 1 && p.mode == MODE_DECODE) {
      const int pp = S.X[b * p.Hq + g * G + hm];
      const int lh = pp >= 1 ? max(pp - p.r + 1, p.sink_f + 1) : p.sink_f + 1;
      lo_mine = lh > lo_mine ? lh : lo_mine;
    }
    float2 o[G][kAPairs], q[G][kAPairs];
    float mrun[G];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      mrun[hh] = kMInit;
#pragma unroll
      for (int i = 0; i < kAPairs; ++i) o[hh][i] = make_float2(0.f, 0.f);
    }
    float m_mine = kMInit, l_mine = 0.f;
    unsigned long long wait_ns = 0;  // traced band waits (kept in a register)

    const int ntiles = tile_count(pc);
    for (int k = 0; k < ntiles; ++k, ++n) {
      const int st = n % kStages;
      const unsigned long long tw = tr_all ? globaltimer() : 0ull;
      const bool ok = wait_use(p, S, n);
      if (tr_all) wait_ns += globaltimer() - tw;
      if (k == 0) {
        stamp(trace, ph ? 13 : 11);
        rotate_query(p, S, st, b, S.u_pos[pc.u]);
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          const float4 x0 = *reinterpret_cast<const float4 *>(S.qrot + hh * kHeadDim + sub * 8);
          const float4 x1 = *reinterpret_cast<const float4 *>(S.qrot + hh * kHeadDim + sub * 8 + 4);
          q[hh][0] = make_float2(x0.x, x0.y);
          q[hh][1] = make_float2(x0.z, x0.w);
          q[hh][2] = make_float2(x1.x, x1.y);
          q[hh][3] = make_float2(x1.z, x1.w);
        }
      }
      const uint8_t *kb = S.stage + (size_t)st * kStageBytes;
      const uint8_t *vb = kb + kStageBytes / 2;
      const int t0 = tile_base(pc, k);  // stage row i holds token t0 + 1 + i
      // partial scores of the group's kATPG tokens for the G heads
      float v[kAV];
#pragma unroll
      for (int tt = 0; tt < kATPG; ++tt) {
        float2 kf[kAPairs];
        row_dims(kb, tt * kAGroups + grp, sub, kf);
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          float2 acc = __fmul2_rn(q[hh][0], kf[0]);
#pragma unroll
          for (int i = 1; i < kAPairs; ++i) acc = __ffma2_rn(q[hh][i], kf[i], acc);
          v[tt * G + hh] = acc.x + acc.y;
        }
      }
      float s = reduce_scores(v, lane);
      const int row_m = ti * kAGroups + grp;
      const int t_m = t0 + row_m + 1;
      // a contiguous tile holds the piece's tokens from its first row on (or
      // nothing, for a refused piece); a paged tile the pages its mask lists
      const int msk = S.mask[st];
      const bool valid = ok && t_m >= lo_mine && t_m <= pc.hi && (PAGED ? ((msk >> (row_m >> 4)) & 1) != 0 : msk != 0);
      s = valid ? s : -INFINITY;
      // lazy running max (per group and head): raised only when a score
      // exceeds it by kLazy
      const float mt = head_max(s);
      if (__any_sync(kFull, mt > m_mine + kLazy)) {
        const float mn_mine = fmaxf(m_mine, mt);
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          const float mn = __shfl_sync(kFull, mn_mine, (lane & 16) | (hh << kAPlain));
          const float f = ex2(mrun[hh] - mn);
          const float2 f2 = make_float2(f, f);
#pragma unroll
          for (int i = 0; i < kAPairs; ++i) o[hh][i] = __fmul2_rn(o[hh][i], f2);
          mrun[hh] = mn;
        }
        l_mine *= ex2(m_mine - mn_mine);
        m_mine = mn_mine;
      }
      const float w = ex2(s - m_mine);
      l_mine += w;
      // rows the piece did not copy hold stale bytes, possibly NaN patterns,
      // and 0 * NaN is NaN: in a partly covered tile they are zeroed
      const bool whole = t0 + kTileTok <= pc.hi &&
                         (PAGED ? t0 + 1 >= pc.lo && msk == (1 << (kTileTok / 16)) - 1 : msk != 0);
#pragma unroll
      for (int tt = 0; tt < kATPG; ++tt) {
        const int row = tt * kAGroups + grp;
        uint4 raw[kALoads];
#pragma unroll
        for (int c = 0; c < kALoads; ++c)
          raw[c] = *reinterpret_cast<const uint4 *>(vb + row * kRowBytes + sub * 8 * (int)sizeof(T) + c * 16);
        if (!whole) {
          const int t = t0 + row + 1;
          const uint32_t vm =
              (PAGED ? t >= pc.lo && t <= pc.hi && ((msk >> (row >> 4)) & 1) != 0 : t <= pc.hi && msk != 0) ? ~0u : 0u;
#pragma unroll
          for (int c = 0; c < kALoads; ++c) raw[c] = make_uint4(raw[c].x & vm, raw[c].y & vm, raw[c].z & vm, raw[c].w & vm);
        }
        float2 vf[kAPairs];
#pragma unroll
        for (int c = 0; c < kALoads; ++c) unpack16x2<T>(raw[c], vf + c * (kAPairs / kALoads));
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
          const float wv = __shfl_sync(kFull, w, (lane & 16) | ((tt * G + hh) << kAPlain));
          const float2 w2 = make_float2(wv, wv);
#pragma unroll
          for (int i = 0; i < kAPairs; ++i) o[hh][i] = __ffma2_rn(w2, vf[i], o[hh][i]);
        }
      }
      release(S, n);
    }
    stamp(trace, ph ? 14 : 12);
    if (tr_all) {
      tr_all[24] = globaltimer();
      tr_all[25] += wait_ns;
    }
    epilogue(p, S, o, mrun, m_mine, l_mine, dst);
    if (ph == 1) stamp(trace, 15);
  }

  // The CTA's kAGroups half-warp states -> one partial summary per head:
  // common maximum, every group rescaled to it, then summed in a fixed order
  // through shared memory.
  __device__ static void epilogue(const StepParams &p, const Smem &S, float2 (&o)[G][kAPairs],
                                  const float (&mrun)[G], float m_mine, float l_mine, float *dst) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, sub = lane & 15;
    const int grp = warp * 2 + (lane >> 4);
    const int idx = sub >> kAPlain, ti = idx / G, hm = idx % G;
    const float l_grp = head_sum(l_mine);  // the group's sum for head hm (all its token slots)
    float mw[G];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) mw[hh] = fmaxf(mrun[hh], __shfl_xor_sync(kFull, mrun[hh], 16));
    if (lane == 0)
#pragma unroll
      for (int hh = 0; hh < G; ++hh) S.red_m[warp * G + hh] = mw[hh];
    consumer_sync();
    float mc[G];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      mc[hh] = S.red_m[hh];
#pragma unroll
      for (int w = 1; w < kWarps; ++w) mc[hh] = fmaxf(mc[hh], S.red_m[w * G + hh]);
    }
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      const float f = ex2(mrun[hh] - mc[hh]);
      const float2 f2 = make_float2(f, f);
#pragma unroll
      for (int i = 0; i < kAPairs; ++i) o[hh][i] = __fmul2_rn(o[hh][i], f2);
    }
    if (ti == 0 && (sub & ((1 << kAPlain) - 1)) == 0) {
      float mcm = mc[0];
#pragma unroll
      for (int hh = 1; hh < G; ++hh) mcm = hm == hh ? mc[hh] : mcm;
      S.red_l[grp * G + hm] = l_grp * ex2(m_mine - mcm);
    }
    {
      float *wr = S.red_o + (size_t)grp * G * kHeadDim + sub * 8;
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        *reinterpret_cast<float4 *>(wr + hh * kHeadDim) = make_float4(o[hh][0].x, o[hh][0].y, o[hh][1].x, o[hh][1].y);
        *reinterpret_cast<float4 *>(wr + hh * kHeadDim + 4) = make_float4(o[hh][2].x, o[hh][2].y, o[hh][3].x, o[hh][3].y);
      }
    }
    consumer_sync();
    // each output element: the kAGroups group states in a fixed order (the
    // next piece's epilogue writes these buffers only after its first
    // barrier, which every thread reaches after these reads)
    float acc[kOutPer];
#pragma unroll
    for (int j = 0; j < kOutPer; ++j) {
      acc[j] = 0.f;
      const int e = tid + j * kConsumers;
      if (e < G * kHeadDim) {
        float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int w2 = 0; w2 < kAGroups; ++w2) part[w2 & 3] += S.red_o[(size_t)w2 * G * kHeadDim + e];
        acc[j] = (part[0] + part[1]) + (part[2] + part[3]);
      }
    }
    griddep_wait();  // the partials live in the scratch workspace (a tail piece may come before the wait)
#pragma unroll
    for (int j = 0; j < kOutPer; ++j) {
      const int e = tid + j * kConsumers;
      if (e < G * kHeadDim) dst[(e / kHeadDim) * kPartStride + e % kHeadDim] = acc[j];
    }
    if (warp == 0) {
      // lane i < kAGroups holds group i's sums; butterfly over the groups
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        float L = lane < kAGroups ? S.red_l[lane * G + hh] : 0.f;
#pragma unroll
        for (int o2 = kAGroups / 2; o2 >= 1; o2 >>= 1) L += __shfl_xor_sync(kFull, L, o2);
        if (lane == hh) {
          dst[hh * kPartStride + kHeadDim] = mc[hh];
          dst[hh * kPartStride + kHeadDim + 1] = L;
        }
      }
    }
  }

  // The CTA's pieces of one kind, in the order both the producer and the
  // consumers walk them: 0 its tail span, 1 its short bands, 2 its
  // long-band span; kind 3 lists (without attention) the units u = c mod P
  // whose merge no band piece triggers: no band piece (the last piece was a
  // tail piece, before the decisions) or no piece at all (no valid length).
  struct PieceIter {
    int kind, it, end;
  };

  // The front sink [1, min(F, m)] of unit u: its length (0 without a sink
  // piece), and the CTA that attends it: with units aligned to CTAs, the
  // first CTA of the unit's group after its tail run (the group's last when
  // the tail takes them all), else u mod P.
  __device__ static int sink_len(const StepParams &p, const Smem &S, int u) {
    if (!SINK || !p.sink_piece) return 0;
    const int64_t m = unit_len(p, S, u);
    if (!len_ok(p, m)) return 0;
    return (int)(m < p.sink_f ? m : p.sink_f);
  }
  __device__ static int sink_cta(const StepParams &p, const Smem &S, int u) {
    const int U = p.B * p.Hkv, P = gridDim.x;
    if (U > P) return u % P;
    const short2 run = S.runA[u];
    const int a = u * P / U, a_next = (u + 1) * P / U;
    const int cand = a + (run.y >= run.x ? run.y - run.x + 1 : 0);
    return cand < a_next ? cand : a_next - 1;
  }
  __device__ static PieceIter piece_iter(const StepParams &p, const Smem &S, int kind) {
    const int U = p.B * p.Hkv, ph = kind == 0 ? 0 : 1;
    PieceIter I;
    I.kind = kind;
    if (kind == 1) {
      short_range(S, &I.it, &I.end);
    } else if (kind == 3) {
      I.it = blockIdx.x;
      I.end = U;
    } else {
      const int64_t g0 = spans(S, ph)[blockIdx.x], g1 = spans(S, ph)[blockIdx.x + 1];
      I.it = g0 < g1 ? unit_of(offs(S, ph), U, g0) : U;
      I.end = U;
    }
    if (SINK && kind == 0 && p.sink_piece) {
      // the sink candidates first: units c, c + P, ..., or, with units
      // aligned to CTAs, the one whose group holds CTA c
      const int P = gridDim.x, c = blockIdx.x;
      I.end = -(I.it + 1);
      I.it = U > P ? c : ((c + 1) * U - 1) / P;
    }
    return I;
  }
  __device__ static bool next_piece(const StepParams &p, const Smem &S, PieceIter &I, Piece &pc) {
    pc.sink = 0;
    if (I.kind == 1) {
      if (I.it >= I.end) return false;
      pc = short_piece(p, S, I.it++);
      return true;
    }
    // kind 0: the CTA's sink pieces come before its tail pieces; while they
    // are looked for, it is the candidate unit and end = -(tail start + 1)
    if (SINK && I.end < 0) {
      const int U = p.B * p.Hkv, P = gridDim.x;
#pragma unroll 1
      for (; I.it < U; I.it += U > P ? P : U) {
        const int u = I.it, n = sink_len(p, S, u);
        if (n > 0 && sink_cta(p, S, u) == (int)blockIdx.x) {
          pc.u = u;
          pc.lo = 1;
          pc.hi = n;
          pc.sink = 1;
          I.it += U > P ? P : U;
          return true;
        }
      }
      I.it = -I.end - 1;
      I.end = U;
    }
    if (I.kind == 3) {
#pragma unroll 1
      for (; I.it < I.end; I.it += gridDim.x) {
        const PieceList L = unit_list(p, S, I.it);
        if (band_pieces(S, L) == 0 &&
            (p.mode == MODE_DECODE || nonempty(S, 0, L.ca0, L.ca0 + L.nt - 1) == 0)) {
          pc.u = I.it;
          pc.lo = 1;
          pc.hi = 0;
          I.it += gridDim.x;
          return true;
        }
      }
      return false;
    }
    const int ph = I.kind == 0 ? 0 : 1;
    if (!find_piece(p, S, ph, I.it, spans(S, ph)[blockIdx.x], spans(S, ph)[blockIdx.x + 1], &pc)) return false;
    I.it = pc.u + 1;
    return true;
  }

  // The consumers' side: attention of each piece, its count, and the merges
  // it completes (one call site each, so the code is inlined once).
  __device__ static void attend_kind(const StepParams &p, const Smem &S, uint32_t &n, int kind) {
    const int U = p.B * p.Hkv, ph = kind == 0 ? 0 : 1;
    PieceIter I = piece_iter(p, S, kind);
    int j0, j1;
    short_range(S, &j0, &j1);
    bool first = kind != 2 || j1 == j0;  // the CTA's first band piece is traced
    Piece pc;
#pragma unroll 1
    while (next_piece(p, S, I, pc)) {
      int act = 2, k = 0;
      if (kind != 3) {
        const size_t slot = kind == 0 ? (size_t)(pc.u + blockIdx.x)
                                      : kind == 1 ? (size_t)pc.u : (size_t)(U + pc.u + blockIdx.x);
        float *dst = SINK && pc.sink ? p.part_s + (size_t)pc.u * G * kPartStride
                             : (ph ? p.part_b : p.part_a) + slot * G * kPartStride;
        attend_piece(p, S, n, ph, pc, dst, first);
        first = false;
        act = piece_count(p, S, pc.u, ph, kind == 1, &k);
      }
      if (act) merge_chain(p, S, pc.u, act, k);
    }
  }

  // ---------------------------------------------------------------------
  // merges
  // ---------------------------------------------------------------------

  // CTAs whose spans meet unit u's segment in phase ph: [*c0, *c1] (empty
  // when *c1 < *c0).
  __device__ static void seg_ctas(const Smem &S, int ph, int u, int *c0, int *c1) {
    const short2 r = (ph ? S.runB : S.runA)[u];
    *c0 = r.x;
    *c1 = r.y;
  }
  // the run of unit u in phase ph, from the offsets and spans
  __device__ static short2 find_run(const Smem &S, int ph, int u) {
    const int64_t *off = offs(S, ph), *span = spans(S, ph);
    if (off[u + 1] <= off[u]) return make_short2(0, -1);
    return make_short2((short)cta_of(span, gridDim.x, off[u]), (short)cta_of(span, gridDim.x, off[u + 1] - 1));
  }

  // Non-empty spans of phase ph among CTAs [c0, c1].
  __device__ static int nonempty(const Smem &S, int ph, int c0, int c1) {
    if (c1 < c0) return 0;
    const int *ne = ph ? S.neB : S.neA;
    return ne[c1 + 1] - ne[c0];
  }

  // The partials a merge reads, in order: nb band entries, then (for a unit)
  // one per CTA of its tail run.  Band entries: the short piece, one per CTA
  // of the long-band run, or, for a run over more than kGroupCtas CTAs, one
  // per CTA group (merged first, each by the CTA that finishes the group's
  // last piece).  A group merge lists the run's CTAs in group k.
  enum { kShort = 0, kCtas = 1, kGroupList = 2 };
  struct PieceList {
    int kind, nb, n;
    int nt;      // tail entries (after the band entries; a sink entry, if any, is last)
    int b0, b1;  // the band entries' CTA range (kCtas) / the whole run (kGroupList)
    int ca0;     // first CTA of the tail run
    int u;
  };
  __device__ static PieceList unit_list(const StepParams &p, const Smem &S, int u) {
    PieceList L;
    int ca1;
    L.u = u;
    seg_ctas(S, 1, u, &L.b0, &L.b1);
    seg_ctas(S, 0, u, &L.ca0, &ca1);
    if (short_band(p, S, u)) {
      L.kind = kShort;
      L.nb = 1;
    } else if (L.b1 - L.b0 + 1 > kGroupCtas) {
      L.kind = kGroupList;
      L.nb = L.b1 / kGroupCtas - L.b0 / kGroupCtas + 1;
    } else {
      L.kind = kCtas;
      L.nb = L.b1 - L.b0 + 1;
    }
    L.nt = ca1 - L.ca0 + 1;
    L.n = L.nb + L.nt + (sink_len(p, S, u) > 0 ? 1 : 0);
    return L;
  }
  __device__ static void group_ctas(const PieceList &L, int k, int *lo, int *hi) {
    *lo = max(L.b0, k * kGroupCtas);
    *hi = min(L.b1, k * kGroupCtas + kGroupCtas - 1);
  }
  __device__ static PieceList group_list(const PieceList &U_, int k) {
    PieceList L = U_;
    L.kind = kCtas;
    group_ctas(U_, k, &L.b0, &L.b1);
    L.nb = L.n = L.b1 - L.b0 + 1;
    L.nt = 0;
    return L;
  }
  // band pieces of the unit (merge inputs made by attention)
  __device__ static int band_pieces(const Smem &S, const PieceList &L) {
    return L.kind == kShort ? 1 : nonempty(S, 1, L.b0, L.b1);
  }
  // what the unit's count must reach: its band entries that exist (pieces,
  // or groups with a piece) and, without a grid barrier before the bands,
  // its tail pieces
  __device__ static int unit_target(const StepParams &p, const Smem &S, const PieceList &L) {
    int n = 0;
    if (L.kind == kGroupList) {
#pragma unroll 1
      for (int k = L.b0 / kGroupCtas; k <= L.b1 / kGroupCtas; ++k) {
        int lo, hi;
        group_ctas(L, k, &lo, &hi);
        n += nonempty(S, 1, lo, hi) > 0;
      }
    } else {
      n = band_pieces(S, L);
    }
    if (p.mode != MODE_DECODE) n += nonempty(S, 0, L.ca0, L.ca0 + L.nt - 1);
    return n;
  }
  __device__ static const float *piece_at(const StepParams &p, const Smem &S, const PieceList &L, int hh, int i) {
    const int U = p.B * p.Hkv, u = L.u;
    if (i < L.nb) {
      if (L.kind == kShort) return p.part_b + ((size_t)u * G + hh) * kPartStride;
      if (L.kind == kCtas) {
        const int c = L.b0 + i;
        if (S.spanB[c] >= S.spanB[c + 1]) return nullptr;
        return p.part_b + ((size_t)(U + u + c) * G + hh) * kPartStride;
      }
      const int k = L.b0 / kGroupCtas + i;
      int lo, hi;
      group_ctas(L, k, &lo, &hi);
      if (nonempty(S, 1, lo, hi) == 0) return nullptr;
      return p.part_g + ((size_t)(u + k) * G + hh) * kPartStride;
    }
    if (SINK && i >= L.nb + L.nt) return p.part_s + ((size_t)u * G + hh) * kPartStride;  // the sink
    const int c = L.ca0 + (i - L.nb);
    if (S.spanA[c] >= S.spanA[c + 1]) return nullptr;
    return p.part_a + ((size_t)(u + c) * G + hh) * kPartStride;
  }

  // Merge of a unit (group < 0) or of CTA group `group` of its long band.
  // The G heads are merged concurrently by kWarps / G warps each, split by
  // dims: every warp of a head goes through the whole list for its slice of
  // the head's dims (lane j holds entry j's pointer, maximum and sum; up to
  // kBatch entries' outputs are in flight at once), so a list of up to
  // kBatch entries costs one trip to L2 and no warp waits for another.  Each class
  // (band, tail) is summed at its maximum over the entries holding tokens.
  // A unit: the cached summary of a hit head with the band state (giving
  // AS_{1:m-r}), then the tail state (giving the output).  A group: the band
  // state, written as a partial like a piece's.  The count the merge
  // answered is cleared for the next launch.
  __device__ static void merge_unit(const StepParams &p, const Smem &S, const PieceList &L, int group) {
    unsigned long long *trace = cta_trace(p);
    const unsigned long long t_in = trace && threadIdx.x == 0 ? globaltimer() : 0ull;
    merge_heads(p, S, L, group);
    if (trace && threadIdx.x == 0) {
      // merge statistics: total time, count, longest merge and its entries
      const unsigned long long dt = globaltimer() - t_in;
      trace[18] += dt;
      trace[19] += 1;
      if (dt > trace[20]) {
        trace[20] = dt;
        trace[21] = (unsigned long long)L.n;
      }
    }
    __syncwarp();
  }

  // N consecutive floats of a partial or ring row (L2, not L1: written by
  // other CTAs), and their store
  template <int N>
  __device__ static void load_dims(const float *src, float (&v)[N]) {
    if constexpr (N == 2) {
      const float2 x = __ldcg(reinterpret_cast<const float2 *>(src));
      v[0] = x.x;
      v[1] = x.y;
    } else {
      v[0] = __ldcg(src);
    }
  }
  template <int N>
  __device__ static void store_dims(float *dst, const float (&v)[N]) {
    if constexpr (N == 2)
      *reinterpret_cast<float2 *>(dst) = make_float2(v[0], v[1]);
    else
      dst[0] = v[0];
  }
  // Log-domain states (base 2): a set of members (m_i, l_i, o_i) combines
  // at the largest m_i among those with l_i > 0, each weighted by
  // 2^(m_i - M).
  // the weight of a member (m, l) in a state at maximum M
  __device__ static float mweight(float m, float l, float M) { return l > 0.f ? ex2(m - M) : 0.f; }

  __device__ static void merge_heads(const StepParams &p, const Smem &S, const PieceList &L, int group) {
    constexpr int kWPH = kWarps / G;         // warps per head
    constexpr int kDW = kHeadDim / kWPH;     // dims of a head per warp
    constexpr int kDL = kDW >= 32 ? kDW / 32 : 1;  // dims per lane
    constexpr int kLanes = kDW / kDL;        // lanes holding dims
    constexpr int kBatch = kDL == 2 ? 10 : 12;  // entries whose outputs a warp asks for at once
    static_assert(kDL == 1 || kDL == 2, "dims per lane");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hh = warp / kWPH, wi = warp % kWPH;
    const int u = L.u, b = u / p.Hkv, g = u - b * p.Hkv;
    const int bh = b * p.Hq + g * G + hh;
    const int n = L.n, nb = L.nb;
    const bool fin = group < 0, decode = p.mode == MODE_DECODE;
    // this lane's dims of the head: [dl, dl + kDL) (lanes past kLanes hold
    // copies of the last lane's, never written)
    const int dl = wi * kDW + min(lane, kLanes - 1) * kDL;
    const bool own = lane < kLanes;
    // Loads here are unconditional, from valid addresses (an empty entry
    // reads a zero partial), so that no instruction waits on their data
    // before it is used.  The cached rectified summary of a hit head:
    bool hit = false;
    float c_lse = 0.f, c_o[kDL];
    if (fin && decode) {
      const int pos = S.X[bh];
      hit = pos >= 1;
      const int64_t slot = (int64_t)bh * p.K + (hit ? pos % p.K : 0);
      c_lse = p.ring_lse[slot];
      load_dims<kDL>(p.ring_o + slot * kHeadDim + dl, c_o);
    }
    // the append: slot pos mod K of the head's rings (the fused append
    // writes it here; otherwise the append kernel does, from staging)
    const int pos = S.u_pos[u];
    const bool app = fin && decode && p.app_o && len_ok(p, pos);
    const int64_t app_slot = (int64_t)bh * p.K + pos % p.K;

    // The whole list for this head, 32 entries at a time (lane j: entry
    // j's pointer, maximum and sum) and up to kBatch outputs in flight:
    // every warp of the head goes through all entries for its dims, so no
    // warp waits for another.  Each class (band, tail) is summed at its
    // maximum over the entries holding tokens.
    float Mb = -INFINITY, Lb = 0.f, Ob[kDL], Mt = -INFINITY, Lt = 0.f, Ot[kDL];
#pragma unroll
    for (int i = 0; i < kDL; ++i) Ob[i] = Ot[i] = 0.f;
#pragma unroll 1
    for (int base = 0; base < n; base += 32) {
      const int cnt = min(32, n - base);
      const float *src = lane < cnt ? piece_at(p, S, L, hh, base + lane) : nullptr;
      if (!src) src = g_zero_partial;
      const float2 ml = __ldcg(reinterpret_cast<const float2 *>(src + kHeadDim));
      const unsigned long long sp = reinterpret_cast<unsigned long long>(src);
      float ov[kBatch][kDL];
#pragma unroll
      for (int k = 0; k < kBatch; ++k)
        load_dims<kDL>(reinterpret_cast<const float *>(__shfl_sync(kFull, sp, k)) + dl, ov[k]);
      const bool band = base + lane < nb;
      float mb = band && ml.y > 0.f ? ml.x : -INFINITY, mt = !band && ml.y > 0.f ? ml.x : -INFINITY;
#pragma unroll
      for (int o2 = 16; o2 >= 1; o2 >>= 1) {
        mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, o2));
        mt = fmaxf(mt, __shfl_xor_sync(kFull, mt, o2));
      }
      // what earlier rounds summed (none in the common case), at the new maxima
      mb = fmaxf(Mb, mb);
      mt = fmaxf(Mt, mt);
      const float rb = mweight(Mb, Lb, mb), rt = mweight(Mt, Lt, mt);
      Lb *= rb;
      Lt *= rt;
#pragma unroll
      for (int i = 0; i < kDL; ++i) {
        Ob[i] *= rb;
        Ot[i] *= rt;
      }
      Mb = mb;
      Mt = mt;
      const float w = mweight(ml.x, ml.y, band ? Mb : Mt);
      const float wb = band ? w : 0.f, wt = band ? 0.f : w;
      float lb = wb * ml.y, lt = wt * ml.y;
#pragma unroll
      for (int o2 = 16; o2 >= 1; o2 >>= 1) {
        lb += __shfl_xor_sync(kFull, lb, o2);
        lt += __shfl_xor_sync(kFull, lt, o2);
      }
      Lb += lb;
      Lt += lt;
#pragma unroll 1
      for (int k0 = 0; k0 < cnt; k0 += kBatch) {
        if (k0 > 0) {
#pragma unroll
          for (int k = 0; k < kBatch; ++k)
            load_dims<kDL>(reinterpret_cast<const float *>(__shfl_sync(kFull, sp, (k0 + k) & 31)) + dl, ov[k]);
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          const int j = (k0 + k) & 31;
          const float xb = __shfl_sync(kFull, wb, j), xt = __shfl_sync(kFull, wt, j);
#pragma unroll
          for (int i = 0; i < kDL; ++i) {
            Ob[i] = fmaf(xb, ov[k][i], Ob[i]);
            Ot[i] = fmaf(xt, ov[k][i], Ot[i]);
          }
        }
      }
    }
    // band: the cached summary (a state of sum 1 at its ln-LSE) with the
    // band state
    const float cm = hit ? c_lse * kLog2e : -INFINITY;
    const float M = fmaxf(cm, Lb > 0.f ? Mb : -INFINITY);
    const float wc = mweight(cm, hit ? 1.f : 0.f, M), wbb = mweight(Mb, Lb, M);
    const float La = (hit ? wc : 0.f) + wbb * Lb;
    float Oa[kDL];
#pragma unroll
    for (int i = 0; i < kDL; ++i) Oa[i] = (hit ? wc * c_o[i] : 0.f) + wbb * Ob[i];
    if (!fin) {
      // the group's partial: the raw state, in a piece partial's layout
      float *dst = p.part_g + ((size_t)(u + group) * G + hh) * kPartStride;
      if (own) store_dims<kDL>(dst + dl, Oa);
      if (wi == 0 && lane == 0) {
        dst[kHeadDim] = M;
        dst[kHeadDim + 1] = La;
      }
    } else {
      if (p.as_o || app) {
        // AS_{1:m-r}, normalised, with its ln-LSE: the rectified summary
        // the ring keeps for position m
        const float inv = La > 0.f ? rcp_approx(La) : 0.f;
        float as[kDL];
#pragma unroll
        for (int i = 0; i < kDL; ++i) as[i] = Oa[i] * inv;
        const float lse = La > 0.f ? (M + lg2_approx(La)) * kLn2 : -INFINITY;
        if (app) {
          // a match at p = m - K reads the slot the append overwrites: every
          // warp of the head has read the cached summary's LSE before the
          // first warp stores the new one (each lane rewrites only the dims
          // it read itself)
          named_sync(2 + hh, kWPH * 32);
          if (own) store_dims<kDL>(p.app_o + app_slot * kHeadDim + dl, as);
          if (wi == 0 && lane == 0) {
            p.app_lse[app_slot] = lse;
            if (hh == 0 && g == 0) p.app_pos[(int64_t)b * p.K + pos % p.K] = pos;
          }
        } else {
          if (own) store_dims<kDL>(p.as_o + (int64_t)bh * kHeadDim + dl, as);
          if (wi == 0 && lane == 0) p.as_lse[bh] = lse;
        }
      }
      // the output: the band state with the tail state
      const float M2 = fmaxf(La > 0.f ? M : -INFINITY, Lt > 0.f ? Mt : -INFINITY);
      const float wa = mweight(M, La, M2), wtt = mweight(Mt, Lt, M2);
      const float L2 = wa * La + wtt * Lt;
      const float inv = L2 > 0.f ? rcp_approx(L2) : 0.f;
      float o[kDL];
#pragma unroll
      for (int i = 0; i < kDL; ++i) o[i] = (wa * Oa[i] + wtt * Ot[i]) * inv;
      if (own) store_dims<kDL>(p.out + (int64_t)bh * kHeadDim + dl, o);
      if (p.out_lse && wi == 0 && lane == 0) p.out_lse[bh] = L2 > 0.f ? (M2 + lg2_approx(L2)) * kLn2 : -INFINITY;
    }
    if (tid == 0) {
      if (fin)
        p.unit_done[u] = 0;
      else
        p.group_done[u + group] = 0;
    }
    consumer_sync();
  }

  // After a piece's partial is written: count it.  Returns what the count
  // completes: 0 nothing, 1 CTA group *k of the unit's long band (merge it
  // first), 2 the unit (every CTA knows how many pieces each unit and group
  // has, so no grid barrier is needed before the merges).  A long-band
  // piece of a two-level unit counts in its CTA group.  A decode step's tail
  // pieces are not counted: they all finish before the grid barrier, which
  // orders them before every merge (so a short band completes its unit).
  __device__ static int piece_count(const StepParams &p, const Smem &S, int u, int ph, bool is_short, int *k) {
    const bool decode = p.mode == MODE_DECODE;
    if (decode && ph == 0) return 0;
    // a short band is its unit's only band piece, and a decode step's tail
    // pieces all finished before the grid barrier: its CTA merges the unit
    // without counting
    if (decode && is_short) return 2;
    *k = blockIdx.x / kGroupCtas;
    // the barrier orders every thread's part of the partial before thread
    // 0's count, whose release makes them visible to the CTA that merges
    consumer_sync();
    if (threadIdx.x == 0) {
      const PieceList L = unit_list(p, S, u);
      int act = 0;
      if (ph == 1 && !is_short && L.kind == kGroupList) {
        int lo, hi;
        group_ctas(L, *k, &lo, &hi);
        const uint32_t old = atom_add_acq_rel_u32(&p.group_done[u + *k], 1u);
        act = (int)(old + 1) == nonempty(S, 1, lo, hi) ? 1 : 0;
      } else {
        const uint32_t old = atom_add_acq_rel_u32(&p.unit_done[u], 1u);
        act = (int)(old + 1) == unit_target(p, S, L) ? 2 : 0;
      }
      *S.last = act;
    }
    consumer_sync();
    return *S.last;
  }

  // The merges a count completed: group k (act 1), which then counts in the
  // unit and may complete it, and the unit (act 2).
  __device__ static void merge_chain(const StepParams &p, const Smem &S, int u, int act, int k) {
    const PieceList Lu = unit_list(p, S, u);
#pragma unroll 1
    while (act) {
      // the other CTAs' partials are visible: thread 0's count acquired
      // them (or the grid barrier ordered them) before a consumer barrier
      merge_unit(p, S, act == 1 ? group_list(Lu, k) : Lu, act == 1 ? k : -1);
      if (act == 2) break;
      // the group partial, ordered by the merge's closing barrier before
      // thread 0's count releases it
      if (threadIdx.x == 0) {
        const uint32_t old = atom_add_acq_rel_u32(&p.unit_done[u], 1u);
        *S.last = (int)(old + 1) == unit_target(p, S, Lu) ? 2 : 0;
      }
      consumer_sync();
      act = *S.last;
    }
  }

  // ---------------------------------------------------------------------

  __device__ static void run(const StepParams &p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int s_mask[kStages];
    __shared__ int s_abort, s_ready, s_last, s_rpar, s_nshort, s_badlen;
    __shared__ uint32_t s_issued;
    __shared__ int64_t s_span[2][kMaxGrid + 1];
    __shared__ int s_ne[2][kMaxGrid + 1];
    __shared__ long long s_short_max, s_band_tot[2], s_scan[kWarps];
    const int n_units = p.B * p.Hkv, n_heads = p.B * p.Hq;
    Smem S;
    S.stage = smem;
    S.qbuf = smem + kOffQ;
    S.full = reinterpret_cast<uint64_t *>(smem + kOffBar);
    S.empty = S.full + kStages;
    S.qrot = reinterpret_cast<float *>(smem + kOffQrot);
    S.red_o = reinterpret_cast<float *>(smem + kOffRedO);
    S.red_l = reinterpret_cast<float *>(smem + kOffRedL);
    S.red_m = reinterpret_cast<float *>(smem + kOffRedM);
    S.X = reinterpret_cast<int32_t *>(smem + kOffX);
    S.offA = reinterpret_cast<int64_t *>(smem + off_units(p.B, p.Hq, p.K));
    S.offB = S.offA + (n_units + 1);
    S.spanA = s_span[0];
    S.spanB = s_span[1];
    S.neA = s_ne[0];
    S.neB = s_ne[1];
    S.scp = S.offB + (n_units + 1);
    S.u_pos = reinterpret_cast<int32_t *>(S.scp + (n_units + 1));
    S.u_s = S.u_pos + n_units;
    S.shortU = S.u_s + n_units;
    S.runA = reinterpret_cast<short2 *>(S.shortU + n_units);
    S.runB = S.runA + n_units;
    S.n_short = &s_nshort;
    S.short_max = &s_short_max;
    S.band_tot = s_band_tot;
    S.scan = s_scan;
    S.rope = p.B <= kRopeTab ? reinterpret_cast<float2 *>(smem + off_rope(p.B, p.Hq, p.Hkv, p.K)) : nullptr;
    S.mask = s_mask;
    S.abort = &s_abort;
    S.ready = &s_ready;
    S.issued = &s_issued;
    S.last = &s_last;
    const bool decode = p.mode == MODE_DECODE;
    const int tid = threadIdx.x;
    unsigned long long *trace = tid < kConsumers ? cta_trace(p) : nullptr;
    if (trace && tid == 0) {
      trace[16] = (unsigned long long)clock64();
      for (int k = 18; k < kTracePoints; ++k) trace[k] = 0;
    }
    stamp(trace, 0);
    if (tid == 0) {
      for (int i = 0; i < kStages; ++i) {
        mbar_init(smem_addr(&S.full[i]), 1);
        mbar_init(smem_addr(&S.empty[i]), kWarps);
      }
      s_abort = 0;
      s_ready = 0;
      s_issued = 0;
      s_badlen = 0;
      // the ring's match state in use: the step count's parity (the previous
      // step on this ring has finished: it is never started early)
      s_rpar = decode ? (int)(*(volatile uint32_t *)p.ring_ctl & 1u) : 0;
      mbar_fence_init();
    }
    __syncthreads();  // the last barrier of all kThreads threads
    S.rpar = s_rpar;
    // The next step kernel on the stream may start its CTAs on the SMs this
    // grid frees.  Until their dependency wait they read only inputs (this
    // launch's queries and lengths, their own layer's rings) and write only
    // shared memory and their own layer's ring state; the host launches them
    // early only when this launch writes none of those (a step on another
    // ring, or full attention).
    griddep_launch_dependents();
    const int n_bh = n_heads;

    if (tid >= kConsumers) {
      producer_warp(p, S);
      return;
    }

#pragma unroll 1
    for (int u = tid; u < n_units; u += kConsumers) {
      S.u_pos[u] = (int32_t)((int64_t)p.pos_base[u / p.Hkv] + p.pos_add);
      S.u_s[u] = p.sink_f + 1;
      if (p.check_len && blockIdx.x == 0 && !len_ok(p, (int64_t)S.u_pos[u] - p.len_sub)) s_badlen = 1;
    }
    if (decode) {
      // every request's length, for the match (X holds the decisions only
      // after the grid barrier)
#pragma unroll 1
      for (int b = tid; b < p.B; b += kConsumers) {
        const int64_t m = (int64_t)p.pos_base[b] + p.pos_add - p.len_sub;
        S.X[b] = m >= 1 && m <= p.max_len ? (int32_t)m : 0;
      }
    }
    if (S.rope && p.rope_mode != MAC_ROPE_NONE) {
      // the rotation angles of every request's query (shared by its heads)
#pragma unroll 1
      for (int i = tid; i < p.B * (kHeadDim / 2); i += kConsumers) {
        const int b = i / (kHeadDim / 2), j = i % (kHeadDim / 2);
        float c, sn;
        rope_angle((int64_t)p.pos_base[b] + p.pos_add, p.rope_f[j], &c, &sn);
        S.rope[i] = make_float2(c, sn);
      }
    }
    consumer_sync();
    layout_tails(p, S);
    if (tid == 0) {
      __threadfence_block();
      *S.ready = 1;  // the producer may copy tail tiles
    }
    stamp(trace, 7);
    uint32_t n = 0;  // stage uses consumed so far (every consumer counts the same sequence)
    // The match, as many chunks as the producer took from the ring's
    // counter, then the tail pieces (every head attends them whatever the
    // match decides): neither needs the scratch workspace (the tail
    // partials' stores wait for the previous kernel), so both may run while
    // the previous kernel on the stream finishes.  Full attention counts
    // every piece at its unit, so it lays out the bands before the first
    // piece and waits at once.
    if (decode) match_phase(p, S, n);
    stamp(trace, 1);
    // From the dependency wait on, the scratch workspace is used: the
    // previous kernel on the stream has finished and its writes are visible.
    auto scratch_ready = [&]() {
      griddep_wait();
      if (tid == 0 && s_badlen) set_status(p.ctl, MAC_DEV_BAD_SEQ_LEN);
    };
    if (!decode) scratch_ready();
    // piece kinds: tails, short bands, long bands, then the merges no piece
    // triggers; the band layout comes before the tails (full attention) or
    // after the match and the decisions (decode): one call site
#pragma unroll 1
    for (int kind = 0; kind < 4; ++kind) {
      if (kind == (decode ? 1 : 0)) {
        if (decode) {
          stamp(trace, 2);
          scratch_ready();
          // the merge counts start from zero, also after a launch that
          // failed with counts left over (no merge runs before the barrier;
          // the host clears them ahead of a full-attention launch)
#pragma unroll 1
          for (int i = blockIdx.x * kConsumers + tid; i < n_units + kGroups; i += gridDim.x * kConsumers) {
            if (i < n_units) p.unit_done[i] = 0u;
            p.group_done[i] = 0u;
          }
          grid_barrier(p, S);  // the minima of every head are final, the tail partials written
          stamp(trace, 10);
          decide(p, S, trace);
          // nobody uses the ring's other copy of the match state in this
          // launch: clear it for the next step on this ring, which uses it
          // (every CTA read the step count before the barrier)
          unsigned long long *next = ring_best(p, S.rpar ^ 1);
#pragma unroll 1
          for (int i = blockIdx.x * kConsumers + tid; i < n_bh; i += gridDim.x * kConsumers) next[i] = 0ull;
          if (blockIdx.x == 0 && tid == 0) {
            *chunk_counter(p, S.rpar ^ 1) = 0u;
            *p.ring_ctl = *p.ring_ctl + 1u;
            atomicAdd(p.ctl + 6, 1u);  // decode launches
          }
        }
        layout_bands(p, S, trace);
        stamp(trace, 3);
      }
      attend_kind(p, S, n, kind);
    }
    stamp(trace, 4);
    if (tid == 0 && *S.abort) {
      // after an abort the producer may have copies in flight into the
      // stages: wait for them, bounded, before the CTA exits
      const long long t0 = clock64();
      while (*S.issued == 0 && clock64() - t0 < (1LL << 30)) {
      }
      const uint32_t nc = *S.issued;
#pragma unroll 1
      for (uint32_t j = nc > (uint32_t)kStages ? nc - kStages : 0u; j < nc; ++j) {
        const uint32_t bar = smem_addr(&S.full[j % kStages]);
        const long long t1 = clock64();
        while (!mbar_try_wait(bar, (j / kStages) & 1u) && clock64() - t1 < (1LL << 30)) {
        }
      }
    }
    __syncwarp();
    stamp(trace, 6);
    if (trace && tid == 0) trace[17] = (unsigned long long)clock64();
    __syncwarp();
  }
};

template <typename T, int G, bool PAGED, bool SINK, bool TRACE>
__global__ void __launch_bounds__(kThreads, 1) step_kernel(const __grid_constant__ StepParams p) {
  Step<T, G, PAGED, SINK, TRACE>::run(p);
}

}  // namespace mac
