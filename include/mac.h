/*
 * mac.h -- C ABI of the MAC-Attention per-step decode-attention library
 * (libmac_gb300.so, hand-written CUDA for GB300 / sm_103a).
 *
 * The method (sources cited per entry point below):
 *   [MAC]  "MAC-Attention: Match-Amend-Complete attention reuse, up to 99% fewer
 *          KV reads in long-context decoding (MLSys 2026)", pinghaoyang.com.cn
 *   [MACS] "MAC-Attention: A Match-Amend-Complete Scheme for Fast and Accurate
 *          Attention Computation (MLSys 2026)", awesome-system-papers summary
 *   [ACSP] "Attention Cache and Sequence Parallelism", shaojiemike.top
 *
 * Conventions shared by every entry point
 *   - Positions are 1-based.  For request b, m = seq_len[b] is the current
 *     length and the K/V of position m is already in the cache: the caller
 *     writes K/V, keys already rotated by RoPE ([ACSP] MHA decode pseudo-code).
 *   - Query head h reads KV head h / (Hq/Hkv) ([ACSP] repeat_kv).
 *   - Every pointer argument is a DEVICE pointer unless stated otherwise; the
 *     caller owns all memory.  The library never allocates device memory.
 *     It owns two CUDA events per ring workspace (created on first use,
 *     destroyed by mac_release_ring).
 *   - Every call is asynchronous on the given stream(s) and returns a status
 *     code: MAC_OK, or a negative MAC_ERR_* for an invalid argument, an
 *     unsupported configuration or a CUDA launch error; nothing was enqueued
 *     when the return value is negative.  Errors that depend on device data
 *     (bad lengths or page ids, a bounded wait that gave up) never fault: the
 *     kernels skip the offending work, write zeros for it, and set bits of a
 *     device status word read by mac_last_status.
 *   - Buffers must be 16-byte aligned (K/V, queries, rings) and do not alias.
 */
#ifndef MAC_H_
#define MAC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes (return values) --------------------------------------- */
#define MAC_OK 0
#define MAC_ERR_INVALID_ARG (-1)   /* NULL pointer, bad size, misaligned buffer */
#define MAC_ERR_UNSUPPORTED (-2)   /* configuration the kernels do not cover */
#define MAC_ERR_CUDA (-3)          /* a CUDA runtime call or launch failed */

/* ---- device status bits (mac_last_status) ------------------------------- */
#define MAC_DEV_BAD_SEQ_LEN 0x1    /* m < 1 or m beyond the cache: request skipped, output 0 */
#define MAC_DEV_BAD_PAGE 0x2       /* page id outside [0, n_pages): its tokens skipped */
#define MAC_DEV_WAIT_TIMEOUT 0x4   /* a bounded wait on a copy gave up: item skipped */
#define MAC_DEV_NONFINITE_Q 0x8    /* non-finite query: treated as a miss */
#define MAC_DEV_BAD_COPY 0x10      /* a copy outside its tile was refused (internal check) */

/* ---- configuration ------------------------------------------------------ */
enum { MAC_BF16 = 0, MAC_F32 = 1 };
/* Threshold reading: [MAC] "Match (2)" accepts ||q~_m - q~_p|| < (1-tau) sqrt(2d)
 * (d=128, tau=0.45 -> 8.8; larger tau is stricter); [MACS] writes
 * tau sqrt(2d).  Both are offered; the first is the default. */
enum { MAC_THR_ONE_MINUS_TAU = 0, MAC_THR_TAU = 1 };
/* RoPE pairing of the query rotation R(m): half-split (j, j+d/2), interleaved
 * (2j, 2j+1), or none.  Frequencies base^(-2j/d), angle (m-1) w_j. */
enum { MAC_ROPE_HALF = 0, MAC_ROPE_INTERLEAVED = 1, MAC_ROPE_NONE = 2 };

typedef struct {
  int32_t batch;       /* B: request slots */
  int32_t n_q_heads;   /* Hq */
  int32_t n_kv_heads;  /* Hkv; Hq/Hkv in {1, 2, 4, 8} */
  int32_t head_dim;    /* d; 128 */
  int32_t ring_k;      /* K: ring capacity = candidate window [m-K, m-1] ([MAC] "Match (3)") */
  int32_t band_r;      /* r: rectification band ([MAC] "Amend"); r >= 0 */
  double tau;          /* match threshold parameter ([MAC] "Match (2)") */
  int32_t thr_mode;    /* MAC_THR_* */
  double rope_base;    /* RoPE base, e.g. 10000 */
  int32_t rope_mode;   /* MAC_ROPE_* */
  int32_t dtype;       /* MAC_BF16 | MAC_F32: element type of queries, ring queries, K, V */
  int32_t page_size;   /* 0 = contiguous K/V; 16 = paged K/V */
  int32_t min_context; /* steps with m < min_context never reuse ([MAC] production defaults) */
  int64_t max_context; /* largest m any call will see; sizes the scratch workspace */
  int32_t front_sink;  /* F >= 0: front-sink isolation ([MAC] "Production version"): tokens
                          [1, F] stay out of the reused summaries (seeded and appended) and
                          are attended exactly at every decode step; 0 = none; negative:
                          MAC_ERR_INVALID_ARG, above 2^30 - 1: MAC_ERR_UNSUPPORTED */
} mac_config;

/* K/V cache.  Contiguous (page_size 0): k, v are [B][Hkv][capacity][d].
 * Paged (page_size 16): k, v are [n_pages][Hkv][16][d] and page_table is
 * [B][max_pages] int32 (device); token t of request b lives in page
 * page_table[b][(t-1)/16], row (t-1)%16. */
typedef struct {
  const void *k;
  const void *v;
  const int32_t *page_table;
  int64_t capacity;  /* contiguous only: tokens per (b, kv-head) block */
  int32_t max_pages; /* paged only */
  int32_t n_pages;   /* paged only: physical pages (bounds check) */
} mac_kv;

/* Byte offsets of the parts of a ring workspace (for inspection/snapshots). */
typedef struct {
  size_t pos;        /* int32 [B][K]: position held by each slot, 0 = empty */
  size_t q;          /* dtype [B][Hq][K][d]: pre-RoPE query ring */
  size_t o;          /* f32 [B][Hq][K][d]: rectified summaries, normalised (S/Z) */
  size_t lse;        /* f32 [B][Hq][K]: their natural-log LSE (running max + ln Z) */
  size_t stage_q;    /* dtype [B][Hq][d]: this step's pre-RoPE query, for the append */
  size_t stage_o;    /* f32 [B][Hq][d]: this step's AS_{1:m-r}, normalised */
  size_t stage_lse;  /* f32 [B][Hq]: its LSE */
  size_t ctl;        /* the running step's match state (GQA groups up to 4): uint32 step
                        count, uint32 [2] chunk counters, uint64 [2][B][Hq] per-head minima
                        (the step count's parity selects the copy in use) */
  size_t total;      /* bytes */
} mac_ring_layout;

/* ---- entry points ------------------------------------------------------- */

/* Workspace sizes for cfg.  ring_bytes: one per layer (the two per-request
 * rings of capacity K, [MAC] "Paper version: K1/K2/K3": a pre-RoPE query
 * ring and a rectified-summary ring with its ln-LSE, plus a small staging
 * area).  scratch_bytes: shared by all calls on one stream (per-head match
 * minima, split-K piece partials, grid-barrier counter, device status word);
 * it must be zero-filled before its first use (mac_init_rings does it).  Its
 * size does not depend on the context length.  Either pointer may be NULL.
 * Returns MAC_ERR_INVALID_ARG / MAC_ERR_UNSUPPORTED for a bad cfg. */
int mac_workspace_size(const mac_config *cfg, size_t *ring_bytes, size_t *scratch_bytes);

/* Offsets of the ring workspace parts for cfg. */
int mac_ring_layout_of(const mac_config *cfg, mac_ring_layout *layout);

/* Reset the rings and scratch; optionally seed them.  q_seed == NULL: every
 * slot is emptied and all requests miss until decode steps fill the rings
 * (requests whose rings are not ready fall back to exact attention, [MAC]
 * "Production version").  q_seed != NULL: [B][Hq][n_seed][d] pre-RoPE queries
 * of positions L-n_seed+1 .. L with L = prompt_len[b] (device int32 [B]);
 * slot p mod K receives position p, its query and the exact rectified
 * summary AS_{1:p-r} of R(p) q_seed over the prompt K/V -- the state exact
 * decoding of those positions would have left ([MACS] "Design trade-offs":
 * prefill stays on the exact path).  n_seed <= K; positions < 1 are skipped.
 * Enqueued on stream (NULL = default stream). */
int mac_init_rings(const mac_config *cfg, void *ring_ws, void *scratch_ws, const void *q_seed,
                   const int32_t *prompt_len, int32_t n_seed, const mac_kv *kv, void *stream);

/* One MAC decode step for all B requests and Hq heads ([MAC] "Paper version:
 * K1/K2/K3", [MACS] "Core method"):
 *   Match     ring L2 nearest neighbour of the pre-RoPE query q_pre[b][h]
 *             (dtype [B][Hq][d]) among slots with position in [m-K, m-1];
 *             hit iff min ||q~_m - q~_c||^2 < thr^2 (thr per cfg.thr_mode,
 *             rounded to fp32); ties go to the most recent position.
 *   Complete  a hit at p attends q_m = R(m) q~_m over [p-r+1, m] only and
 *             merges it in log domain with the cached summary AS_{1:p-r};
 *             a miss attends over [1, m] (split-K full attention).
 *   Append    on stream_aux after an event: slot m mod K <- (m, q~_m,
 *             AS_{1:m-r}), where AS_{1:m-r} = cached part (+) fresh tokens up
 *             to m-r (the rectified summary; the band and tail are
 *             accumulated separately, so no log-domain subtraction is needed).
 * out: f32 [B][Hq][d] attention output.  match_pos: int32 [B][Hq] matched
 * position, -1 on a miss (may be NULL).  stream_aux NULL: the step kernel
 * writes the rings' slot itself once it has merged a head (the match has
 * read the rings before that), so there is no second kernel and no event.
 * stream_aux == stream_main: the append kernel runs on stream_main after the
 * step.  Another stream: the append kernel runs there after an event, and
 * the next step on the same ring_ws makes stream_main wait for it; a
 * captured CUDA graph must then call mac_join_aux before its capture ends.
 * The three give bitwise identical rings and outputs. */
int mac_decode_step(const mac_config *cfg, void *ring_ws, void *scratch_ws, const void *q_pre,
                    const int32_t *seq_len, const mac_kv *kv, float *out, int32_t *match_pos,
                    void *stream_main, void *stream_aux);

/* Exact split-K decode attention over [1, m] for every (b, h): the miss
 * fallback as a call of its own ([MAC] "Match (1)": a miss reproduces full
 * attention; [ACSP] MHA decode).  The query is rotated by R(m).  out: f32
 * [B][Hq][d]; lse: f32 [B][Hq] natural-log softmax denominator, or NULL.
 * Uses the same chunking and merge order as a decode step in which every
 * head misses, so such a step's output is bitwise equal to this call's; a
 * missing head in a step where others hit attends the same tokens with a
 * chunking that depends on the other units' bands (equal to rounding).  The
 * config's front_sink is ignored (attention over [1, m] is exact either way;
 * with F > 0 a decode step's miss equals this call to rounding). */
int mac_full_attention(const mac_config *cfg, void *scratch_ws, const void *q_pre,
                       const int32_t *seq_len, const mac_kv *kv, float *out, float *lse,
                       void *stream);

/* Largest scratch workspace mac_full_attention_noalloc can use (16 MiB). */
#define MAC_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/* mac_full_attention without a caller-provided scratch workspace.  (The
 * pages have no counterpart; this is a packaging variant.)  For callers that
 * cannot allocate device memory: code whose device memory is owned by
 * another allocator it may not call into, code that must not trigger the
 * device-wide synchronisation cudaMalloc can cause, or code running under a
 * fixed memory budget decided at start-up.  The scratch lives in a 16 MiB
 * array compiled into this library (MAC_NOALLOC_SCRATCH_BYTES); every GPU
 * that loads the library holds that array until the process exits.
 *   - Same arguments and results as mac_full_attention, minus scratch_ws.
 *   - Returns MAC_ERR_UNSUPPORTED, without enqueueing anything, when the
 *     configuration's scratch (mac_workspace_size) exceeds
 *     MAC_NOALLOC_SCRATCH_BYTES.
 *   - Allocates nothing: no cudaMalloc/cudaFree and no allocating library
 *     call.  The first call on a device looks up the array's device address
 *     (once per device, with that device current); make that first call
 *     before any stream capture.
 *   - Every call on a device shares the one array.  Each call clears the
 *     array's counters on its stream before launching, so calls on one
 *     stream are fine; calls that overlap on the GPU (different streams, or
 *     different host threads without ordering) race on the array and give
 *     wrong results.  The device status word of these calls is cleared by
 *     the next call and is not readable through mac_last_status. */
int mac_full_attention_noalloc(const mac_config *cfg, const void *q_pre, const int32_t *seq_len,
                               const mac_kv *kv, float *out, float *lse, void *stream);

/* Make stream_main wait for the last append enqueued on ring_ws (no-op if
 * none is pending).  Needed before ending a stream capture that used a
 * separate aux stream. */
int mac_join_aux(void *ring_ws, void *stream_main);

/* Ready gate ([MAC] "Production version": request state gated so that a
 * captured CUDA graph stays valid).  reset_flags: device int32 [B].  For
 * every request b whose flag is non-zero, its rings start over empty: no
 * slot holds a position any more, so its next decode step has no match
 * candidate, misses on every head and attends [1, m] exactly, and the
 * appends of its next steps refill the rings.  The flags are read and
 * cleared on the device, on `stream`, after any append still pending on an
 * auxiliary stream for ring_ws; the call can be captured into a graph and
 * the caller sets flags between replays (a new request in a reused slot,
 * a request whose cache was rewritten).  Returns MAC_ERR_INVALID_ARG for a
 * null or misaligned pointer; the flags' values are not checked. */
int mac_reset_requests(const mac_config *cfg, void *ring_ws, int32_t *reset_flags, void *stream);

/* Test hook for the bounded waits (no counterpart on the pages): the next
 * step kernel launched by the calling thread gives every wait (a stage's
 * copy, a flag, the grid barrier, a piece count) `cycles` SM cycles instead
 * of about a second, and, if withhold_use >= 0, never issues the copy of
 * that stage use (per CTA in the span kernel, per warp in the ring kernel),
 * so the wait for it runs out: the kernel sets MAC_DEV_WAIT_TIMEOUT, stops
 * its work, lets its other copies land and returns.  The launch's outputs
 * are then undefined; its scratch workspace must be cleared (or replaced)
 * before the next launch.  1 <= cycles <= 2^31, withhold_use >= -1; the
 * hook clears itself. */
int mac_test_wait_budget(int64_t cycles, int32_t withhold_use);

/* Destroy the events the library keeps for ring_ws (call before freeing it). */
int mac_release_ring(void *ring_ws);

/* Synchronise stream, copy the device status word (MAC_DEV_* bits, 0 = clean)
 * to *device_status (host pointer) and clear it. */
int mac_last_status(const mac_config *cfg, void *scratch_ws, int32_t *device_status,
                    void *stream);

/* Profiling hook (no counterpart on the pages): the next mac_decode_step
 * issued by the calling thread records these CUDA events (cudaEvent_t
 * handles, each may be NULL): before and after the step kernel (match and
 * attention) on stream_main, and after the append kernel on the stream it
 * runs on; then the hook clears itself.  Lets a caller time the kernels on
 * the stream they run on, also inside a captured graph. */
int mac_set_phase_events(void *before_step, void *after_step, void *after_append);

/* Profiling hook (no counterpart on the pages): the next step kernel
 * launched by the calling thread (decode step or full attention) writes, per
 * CTA, MAC_TRACE_POINTS uint64 %globaltimer stamps (ns) into device_buffer
 * [grid][MAC_TRACE_POINTS]:
 *    0 start            1 end of the match       2 end of the tail pieces
 *    3 bands laid out   4 end of the band pieces and merges
 *    5 decisions read   6 end              7 tail layout published
 *    8 first match chunk arrived   9 producer: short-band tiles issued
 *   10 after the grid barrier
 *   11/12 first tail piece: first tile arrived / tiles done
 *   13/14 first band piece: first tile arrived / tiles done
 *   15 first band piece's partial written
 *   16/17 the SM's clock64() at start / end (cycles; with 0 and 6 they give
 *         the SM clock during the launch)
 *   18/19 time spent merging units (ns) / units merged
 *   20/21 the longest merge (ns) / its pieces
 *   22/23 band tokens / band pieces the CTA attended
 *   24 last band piece's tiles done   25 time spent waiting for band tiles (ns)
 *   26/27 producer: short-band list seen / long-band layout published
 *   28/29 time spent waiting for match chunks (ns) / match chunks scanned
 *   30/31 producer: first match copies issued / tail layout seen
 * Configurations with Hq/Hkv = 8 run the ring kernel (every warp feeds its
 * own stage ring; no producer warp), whose stamps are:
 *    0 start            1 warp 0's window tiles and match items done
 *    2 after the grid barrier         3 decisions and long bands laid out
 *    4 boundary pieces and hit merges done   5 long bands done
 *    6 end              7 the CTA's exit
 *   13/19 warps 0 / 1: owner merge's list read   14/15 owner merge's
 *         states written / combined  18 owner merge start
 *   16/17 the SM's clock64() at start / end
 * Stamps of phases a launch does not run are left as they were.  The span
 * kernel's stamps are compiled into one instantiation only, bf16 K/V without
 * a front sink, which the launch then runs; other span-kernel launches leave
 * the buffer as it was.  The buffer must hold MAC_TRACE_POINTS * (number of
 * SMs) uint64.  The hook clears itself. */
#define MAC_TRACE_POINTS 32
int mac_set_trace(void *device_buffer);

/* Static string for a MAC_OK / MAC_ERR_* code. */
const char *mac_status_string(int code);

/* Squared match threshold the kernels compare against (fp64 formula rounded
 * once to fp32), for reporting. */
float mac_threshold_sq(const mac_config *cfg);

#ifdef __cplusplus
}
#endif
#endif /* MAC_H_ */
