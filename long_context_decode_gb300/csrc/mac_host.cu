// mac_host.cu -- the C ABI of libmac_gb300 (declared in include/mac.h):
// argument checks, workspace layouts, the per-ring event pair that orders
// the rectify-append on the aux stream, and the kernel launch sequences.
#include <math.h>
#include <string.h>

#include <mutex>
#include <unordered_map>

#include "mac_common.cuh"

using namespace mac;

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int elem_size(const mac_config *c) { return c->dtype == MAC_F32 ? 4 : 2; }

int validate(const mac_config *c) {
  if (!c) return MAC_ERR_INVALID_ARG;
  if (c->batch < 1 || c->n_q_heads < 1 || c->n_kv_heads < 1 || c->ring_k < 1 || c->band_r < 0 ||
      c->max_context < 1 || c->min_context < 0 || !(c->rope_base > 0.0) || !isfinite(c->tau))
    return MAC_ERR_INVALID_ARG;
  if (c->n_q_heads % c->n_kv_heads != 0) return MAC_ERR_INVALID_ARG;
  const int G = c->n_q_heads / c->n_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return MAC_ERR_UNSUPPORTED;
  if (c->head_dim != kHeadDim) return MAC_ERR_UNSUPPORTED;
  if (c->dtype != MAC_BF16 && c->dtype != MAC_F32) return MAC_ERR_INVALID_ARG;
  if (c->page_size != 0 && c->page_size != 16) return MAC_ERR_UNSUPPORTED;
  if (c->thr_mode != MAC_THR_ONE_MINUS_TAU && c->thr_mode != MAC_THR_TAU) return MAC_ERR_INVALID_ARG;
  if (c->rope_mode < MAC_ROPE_HALF || c->rope_mode > MAC_ROPE_NONE) return MAC_ERR_INVALID_ARG;
  if ((int64_t)c->batch * c->n_kv_heads > kMaxUnits) return MAC_ERR_UNSUPPORTED;
  if ((int64_t)c->batch * c->n_q_heads > kMaxHeads) return MAC_ERR_UNSUPPORTED;
  if (c->max_context > 0x7fffffffLL - 1) return MAC_ERR_UNSUPPORTED;
  if (c->front_sink < 0) return MAC_ERR_INVALID_ARG;
  if (c->front_sink > 0x3fffffff) return MAC_ERR_UNSUPPORTED;  // kept clear of 32-bit overflow
  return MAC_OK;
}

mac_ring_layout ring_layout(const mac_config *c) {
  const size_t B = c->batch, H = c->n_q_heads, K = c->ring_k, d = c->head_dim;
  const size_t es = elem_size(c);
  mac_ring_layout L;
  size_t off = 0;
  L.pos = off;       off = align_up(off + B * K * 4, 256);
  L.q = off;         off = align_up(off + B * H * K * d * es, 256);
  L.o = off;         off = align_up(off + B * H * K * d * 4, 256);
  L.lse = off;       off = align_up(off + B * H * K * 4, 256);
  L.stage_q = off;   off = align_up(off + B * H * d * es, 256);
  L.stage_o = off;   off = align_up(off + B * H * d * 4, 256);
  L.stage_lse = off; off = align_up(off + B * H * 4, 256);
  L.ctl = off;       off = align_up(off + 16 + 2 * B * H * 8, 256);
  L.total = off;
  return L;
}

// The step kernel of a configuration: the span kernel for GQA groups of up
// to four query heads, the ring kernel for groups of eight.
bool ring_kernel(const mac_config *c) { return c->n_q_heads / c->n_kv_heads == 8; }

// Ring kernel: tiles per unit of a launch (window and tail, plus the front
// sink when the launch attends it: decode steps with F > 0).
TileCounts launch_tiles(const mac_config *c, bool sink_piece) {
  return ring::tile_counts(c->ring_k, c->band_r, c->max_context, sink_piece ? c->front_sink : 0, elem_size(c));
}

// Everything before `parts` must start at zero (the status word, the
// counters, the per-head minima and the per-unit piece counts); the
// partials need no clearing.  A clean launch leaves it so for the next one.
ScratchLayout scratch_layout(const mac_config *c) {
  const size_t B = c->batch, H = c->n_q_heads, U = (size_t)c->batch * c->n_kv_heads;
  const size_t G = c->n_q_heads / c->n_kv_heads;
  const size_t part = G * kPartStride * 4;  // bytes of one (piece, all heads) partial
  ScratchLayout S = {};
  size_t off = 0;
  S.ctl = off;         off = align_up(off + 64 * 4, 256);
  S.best = off;        off = align_up(off + 2 * B * H * 8, 256);
  S.unit_done = off;   off = align_up(off + 2 * U * 4, 256);
  S.group_done = off;  off = align_up(off + 2 * (U + kGroups) * 4, 256);
  S.parts = off;
  if (ring_kernel(c)) {
    const size_t nt = (size_t)launch_tiles(c, true).nt;
    S.part_w = off;    off = align_up(off + U * nt * part, 256);
    S.part_c = off;    off = align_up(off + (U + kMaxGrid) * part, 256);
    S.part_g = off;    off = align_up(off + (U + kGroups) * part, 256);
    S.part_x = off;    off = align_up(off + (size_t)kMaxGrid * ring::kWarps * part, 256);
  } else {
    const size_t slots = U + kMaxGrid;
    S.part_a = off;    off = align_up(off + slots * part, 256);
    S.part_b = off;    off = align_up(off + (U + slots) * part, 256);
    S.part_g = off;    off = align_up(off + (U + kGroups) * part, 256);
    S.part_s = off;    off = align_up(off + U * part, 256);
  }
  S.total = off;
  return S;
}

float threshold_sq(const mac_config *c) {
  const double f = (c->thr_mode == MAC_THR_TAU) ? c->tau : (1.0 - c->tau);
  const double thr = f * sqrt(2.0 * (double)c->head_dim);
  return (float)(thr * thr);
}

float q_scale(const mac_config *c) { return (float)(1.4426950408889634 / sqrt((double)c->head_dim)); }

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

int check_kv(const mac_config *c, const mac_kv *kv) {
  if (!kv || !kv->k || !kv->v || !aligned16(kv->k) || !aligned16(kv->v)) return MAC_ERR_INVALID_ARG;
  if (c->page_size == 0) {
    if (kv->capacity < 1) return MAC_ERR_INVALID_ARG;
  } else {
    if (!kv->page_table || kv->max_pages < 1 || kv->n_pages < 1) return MAC_ERR_INVALID_ARG;
  }
  return MAC_OK;
}

KvView kv_view(const mac_config *c, const mac_kv *kv) {
  KvView v;
  v.k = kv->k;
  v.v = kv->v;
  v.page_table = kv->page_table;
  v.paged = c->page_size != 0;
  v.capacity = v.paged ? (int64_t)kv->max_pages * c->page_size : kv->capacity;
  v.max_pages = kv->max_pages;
  v.n_pages = kv->n_pages;
  return v;
}

// Largest length the kernels accept: within the cache and within the
// max_context the scratch was sized for.
int64_t max_len(const mac_config *c, const KvView &v) {
  return v.capacity < c->max_context ? v.capacity : c->max_context;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

int step_occupancy(const mac_config *c) {
  const int G = c->n_q_heads / c->n_kv_heads, U = c->batch * c->n_kv_heads;
  const bool paged = c->page_size != 0, f32 = c->dtype == MAC_F32;
  if (ring_kernel(c)) return f32 ? ring::occupancy_f32_g8(paged, U, c->batch) : ring::occupancy_bf16_g8(paged, U, c->batch);
  const int B = c->batch, Hq = c->n_q_heads, Hkv = c->n_kv_heads, K = c->ring_k;
  int per_sm = f32 ? step_occupancy_f32(G, paged, B, Hq, Hkv, K) : step_occupancy_bf16(G, paged, B, Hq, Hkv, K);
  if (c->front_sink > 0) {  // the decode steps launch the sink kernels: the grid must fit both
    const int s = f32 ? step_occupancy_f32_sink(G, paged, B, Hq, Hkv, K) : step_occupancy_bf16_sink(G, paged, B, Hq, Hkv, K);
    per_sm = s < per_sm ? s : per_sm;
  }
  return per_sm;
}

// Persistent grid: as many CTAs as can be resident at once (one per SM), at
// most kMaxGrid (the partial slots are sized for that many).
int step_grid(const mac_config *c) {
  const int per_sm = step_occupancy(c);
  if (per_sm < 1) return 0;
  const int grid = num_sms() * per_sm;
  return grid < kMaxGrid ? grid : kMaxGrid;
}

cudaError_t launch_step(StepParams p, const mac_config *c, cudaStream_t s);

// Common part of every step launch: shapes, constants, K/V, scratch.
StepParams step_params(const mac_config *c, const ScratchLayout &S, uint8_t *scratch,
                       const mac_kv *kv, int mode) {
  StepParams a;
  memset(&a, 0, sizeof a);
  a.mode = mode;
  a.check_len = 1;
  a.B = c->batch;
  a.Hq = c->n_q_heads;
  a.Hkv = c->n_kv_heads;
  a.G = c->n_q_heads / c->n_kv_heads;
  a.K = c->ring_k;
  a.r = c->band_r;
  a.min_context = c->min_context;
  a.thr2 = threshold_sq(c);
  a.q_scale = q_scale(c);
  a.rope_mode = c->rope_mode;
  a.kv = kv_view(c, kv);
  a.max_len = max_len(c, a.kv);
  a.q_stride = c->head_dim;
  for (int j = 0; j < kHeadDim / 2; ++j)
    a.rope_f[j] = (unsigned long long)ldexp(
        pow(c->rope_base, -2.0 * (double)j / (double)c->head_dim) / 6.283185307179586, 64);
  a.ctl = (uint32_t *)(scratch + S.ctl);
  a.best = (unsigned long long *)(scratch + S.best);
  a.unit_done = (uint32_t *)(scratch + S.unit_done);
  a.group_done = (uint32_t *)(scratch + S.group_done);
  a.part_g = (float *)(scratch + S.part_g);
  if (ring_kernel(c)) {
    a.part_w = (float *)(scratch + S.part_w);
    a.part_c = (float *)(scratch + S.part_c);
    a.part_x = (float *)(scratch + S.part_x);
  } else {
    a.part_a = (float *)(scratch + S.part_a);
    a.part_b = (float *)(scratch + S.part_b);
    a.part_s = (float *)(scratch + S.part_s);
  }
  a.tc = launch_tiles(c, false);
  return a;
}

AppendParams append_params(const mac_config *c, const mac_ring_layout &R, uint8_t *ring,
                           const StepParams &sp) {
  AppendParams q;
  memset(&q, 0, sizeof q);
  q.B = c->batch;
  q.Hq = c->n_q_heads;
  q.K = c->ring_k;
  q.pos_base = sp.pos_base;
  q.pos_add = sp.pos_add;
  q.capacity = sp.max_len;
  q.q_stride = c->head_dim;
  q.src_o = (const float *)(ring + R.stage_o);
  q.src_lse = (const float *)(ring + R.stage_lse);
  q.ring_pos = (int32_t *)(ring + R.pos);
  q.ring_q = ring + R.q;
  q.ring_o = (float *)(ring + R.o);
  q.ring_lse = (float *)(ring + R.lse);
  return q;
}

// ---- per-ring events: the append of step n on stream_aux must finish before
// step n+1 on the same ring reads or rewrites the rings ([MAC] K3 runs on an
// auxiliary stream with a single event dependency).
struct RingEvents {
  cudaEvent_t main_done = nullptr, aux_done = nullptr;
  bool pending = false;
  unsigned long long capture_id = 0;
  int device = -1;
};
std::mutex g_mu;
std::unordered_map<void *, RingEvents> g_rings;

// The last library launch on each stream, as far as an early start of the
// next step kernel goes: the ring a fused decode step wrote, or kNoRing
// after full attention (which writes no ring); absent or null after
// anything else (an append kernel, a reset, ring seeding, a step with
// timing events), after which the next step kernel waits as usual.  A step
// kernel's early part reads its queries, its lengths and its own layer's
// rings, so it may start early after a step that wrote another ring.
std::unordered_map<cudaStream_t, const void *> g_last_launch;
const char kNoRingTag = 0;
const void *const kNoRing = &kNoRingTag;

// Records `writes` as the stream's last launch; returns whether a step
// kernel whose early part reads ring `reads` (null: none) may start early.
bool note_launch(cudaStream_t s, const void *reads, const void *writes) {
  std::lock_guard<std::mutex> lk(g_mu);
  const void *prev = nullptr;
  auto it = g_last_launch.find(s);
  if (it != g_last_launch.end()) prev = it->second;
  g_last_launch[s] = writes;
  return prev != nullptr && (reads == nullptr || prev != reads);
}

unsigned long long capture_id_of(cudaStream_t s) {
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  unsigned long long id = 0;
  if (cudaStreamGetCaptureInfo(s, &st, &id) != cudaSuccess) return 0;
  return st == cudaStreamCaptureStatusActive ? id : 0;
}

// Scratch of mac_full_attention_noalloc: a fixed array inside the library,
// for callers that cannot allocate device memory.  Host code must not pass
// the symbol itself to a kernel (on the host it names a host-side stand-in);
// noalloc_scratch() returns its device address.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MAC_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[256] = {nullptr};  // per device, looked up once

// Device address of g_noalloc_scratch on the current device (nullptr on error).
void *noalloc_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 256) return nullptr;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
    g_noalloc_ptr[dev] = p;
  }
  return g_noalloc_ptr[dev];
}

// events armed by mac_set_phase_events for this thread's next decode step
thread_local cudaEvent_t t_phase[3] = {nullptr, nullptr, nullptr};
// trace buffer armed by mac_set_trace for this thread's next step kernel
thread_local unsigned long long *t_trace = nullptr;
// run-out test knob armed by mac_test_wait_budget for this thread's next
// step kernel (0: the default budget)
thread_local long long t_wait_limit = 0;
thread_local int t_withhold = -1;
constexpr long long kWaitLimit = 1LL << 31;  // about a second of SM cycles

cudaError_t launch_step(StepParams p, const mac_config *c, cudaStream_t s) {
  const int grid = step_grid(c);
  if (grid < 1) return cudaErrorInvalidValue;
  p.trace = t_trace;
  t_trace = nullptr;
  p.wait_limit = t_wait_limit > 0 ? t_wait_limit : kWaitLimit;
  p.withhold = t_withhold;
  t_wait_limit = 0;
  t_withhold = -1;
  const bool f32 = c->dtype == MAC_F32;
  if (ring_kernel(c)) {
    p.tc = launch_tiles(c, p.sink_piece != 0);
    return f32 ? ring::launch_f32_g8(p, grid, s) : ring::launch_bf16_g8(p, grid, s);
  }
  if (p.mode == MODE_FULL) {
    // Full attention counts pieces into its merges without a grid barrier
    // before them, so it cannot clear counts a failed launch left behind
    // (a decode step clears them before its barrier): they are cleared
    // here, ahead of it on the stream.
    const ScratchLayout S = scratch_layout(c);
    const cudaError_t e = cudaMemsetAsync(p.unit_done, 0, S.parts - S.unit_done, s);
    if (e != cudaSuccess) return e;
  }
  if (p.sink_piece) return f32 ? launch_step_f32_sink(p, grid, s) : launch_step_bf16_sink(p, grid, s);
  if (p.trace && !f32) return launch_step_bf16_trace(p, grid, s);  // the only traced instantiation
  return f32 ? launch_step_f32(p, grid, s) : launch_step_bf16(p, grid, s);
}

// Inside a stream capture the record becomes an event-record node of the
// graph (timestamped at replay), not a capture-time dependency marker.
cudaError_t record_phase(int i, cudaStream_t s) {
  if (!t_phase[i]) return cudaSuccess;
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &st);
  if (e == cudaSuccess)
    e = st == cudaStreamCaptureStatusActive
            ? cudaEventRecordWithFlags(t_phase[i], s, cudaEventRecordExternal)
            : cudaEventRecord(t_phase[i], s);
  t_phase[i] = nullptr;
  return e;
}

}  // namespace

extern "C" {

int mac_workspace_size(const mac_config *cfg, size_t *ring_bytes, size_t *scratch_bytes) {
  int v = validate(cfg);
  if (v != MAC_OK) return v;
  if (ring_bytes) *ring_bytes = ring_layout(cfg).total;
  if (scratch_bytes) *scratch_bytes = scratch_layout(cfg).total;
  return MAC_OK;
}

int mac_ring_layout_of(const mac_config *cfg, mac_ring_layout *layout) {
  int v = validate(cfg);
  if (v != MAC_OK) return v;
  if (!layout) return MAC_ERR_INVALID_ARG;
  *layout = ring_layout(cfg);
  return MAC_OK;
}

float mac_threshold_sq(const mac_config *cfg) {
  if (validate(cfg) != MAC_OK) return NAN;
  return threshold_sq(cfg);
}

const char *mac_status_string(int code) {
  switch (code) {
    case MAC_OK: return "ok";
    case MAC_ERR_INVALID_ARG: return "invalid argument";
    case MAC_ERR_UNSUPPORTED: return "unsupported configuration";
    case MAC_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

int mac_init_rings(const mac_config *cfg, void *ring_ws, void *scratch_ws, const void *q_seed,
                   const int32_t *prompt_len, int32_t n_seed, const mac_kv *kv, void *stream) {
  int v = validate(cfg);
  if (v != MAC_OK) return v;
  if (!ring_ws || !scratch_ws || !aligned16(ring_ws) || !aligned16(scratch_ws))
    return MAC_ERR_INVALID_ARG;
  if (q_seed && (!prompt_len || !kv || n_seed < 1 || n_seed > cfg->ring_k || !aligned16(q_seed)))
    return MAC_ERR_INVALID_ARG;
  if (q_seed && (v = check_kv(cfg, kv)) != MAC_OK) return v;
  cudaStream_t s = (cudaStream_t)stream;
  note_launch(s, nullptr, nullptr);  // seeding writes the ring: the next step waits
  const mac_ring_layout R = ring_layout(cfg);
  const ScratchLayout S = scratch_layout(cfg);
  uint8_t *ring = (uint8_t *)ring_ws, *scr = (uint8_t *)scratch_ws;
  if (cudaMemsetAsync(ring + R.pos, 0, (size_t)cfg->batch * cfg->ring_k * 4, s) != cudaSuccess ||
      cudaMemsetAsync(ring + R.ctl, 0, R.total - R.ctl, s) != cudaSuccess ||
      cudaMemsetAsync(scr, 0, S.parts, s) != cudaSuccess)
    return MAC_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_rings.find(ring_ws);
    if (it != g_rings.end()) it->second.pending = false;
  }
  if (!q_seed) return MAC_OK;

  // seed i: position p = L - n_seed + 1 + i, exact summary over [1, p - r]
  // of R(p) q_seed[.., i, ..] (the full-attention path), then appended;
  // with a front sink F the summary covers [F+1, p - r]
  StepParams sp = step_params(cfg, S, scr, kv, MODE_FULL);
  sp.sink_f = cfg->front_sink;
  sp.check_len = 0;  // summary lengths p - r may be < 1 (empty summaries)
  sp.pos_base = prompt_len;
  sp.len_sub = cfg->band_r;
  sp.q = q_seed;
  sp.q_stride = (int64_t)n_seed * cfg->head_dim;
  sp.out = (float *)(ring + R.stage_o);
  sp.out_lse = (float *)(ring + R.stage_lse);
  for (int i = 0; i < n_seed; ++i) {
    sp.pos_add = -n_seed + 1 + i;
    sp.q_offset = (int64_t)i * cfg->head_dim;
    AppendParams ap = append_params(cfg, R, ring, sp);
    ap.q_src = q_seed;
    ap.q_stride = sp.q_stride;
    ap.q_offset = sp.q_offset;
    if (launch_step(sp, cfg, s) != cudaSuccess || launch_append(ap, cfg->dtype, s) != cudaSuccess)
      return MAC_ERR_CUDA;
  }
  return MAC_OK;
}

int mac_decode_step(const mac_config *cfg, void *ring_ws, void *scratch_ws, const void *q_pre,
                    const int32_t *seq_len, const mac_kv *kv, float *out, int32_t *match_pos,
                    void *stream_main, void *stream_aux) {
  int v = validate(cfg);
  if (v != MAC_OK) return v;
  if (!ring_ws || !scratch_ws || !q_pre || !seq_len || !out || !aligned16(ring_ws) ||
      !aligned16(scratch_ws) || !aligned16(q_pre) || !aligned16(out))
    return MAC_ERR_INVALID_ARG;
  if ((v = check_kv(cfg, kv)) != MAC_OK) return v;
  cudaStream_t sm = (cudaStream_t)stream_main;
  cudaStream_t sa = stream_aux ? (cudaStream_t)stream_aux : sm;
  const bool use_aux = sa != sm;
  const bool fused = stream_aux == nullptr;  // the step kernel appends itself
  const mac_ring_layout R = ring_layout(cfg);
  const ScratchLayout S = scratch_layout(cfg);
  uint8_t *ring = (uint8_t *)ring_ws, *scr = (uint8_t *)scratch_ws;
  const unsigned long long cap_id = capture_id_of(sm);

  RingEvents *ev = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    RingEvents &e = g_rings[ring_ws];
    if (use_aux && !e.main_done) {
      cudaGetDevice(&e.device);
      if (cudaEventCreateWithFlags(&e.main_done, cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&e.aux_done, cudaEventDisableTiming) != cudaSuccess)
        return MAC_ERR_CUDA;
    }
    if (e.pending && e.capture_id == cap_id) {
      if (cudaStreamWaitEvent(sm, e.aux_done, 0) != cudaSuccess) return MAC_ERR_CUDA;
    }
    e.pending = false;
    ev = &e;
  }

  StepParams sp = step_params(cfg, S, scr, kv, MODE_DECODE);
  sp.sink_f = cfg->front_sink;
  sp.sink_piece = cfg->front_sink > 0;
  sp.pos_base = seq_len;
  sp.q = q_pre;
  sp.ring_pos = (const int32_t *)(ring + R.pos);
  sp.ring_q = ring + R.q;
  sp.ring_o = (const float *)(ring + R.o);
  sp.ring_lse = (const float *)(ring + R.lse);
  sp.stage_q = ring + R.stage_q;
  sp.ring_ctl = (uint32_t *)(ring + R.ctl);
  sp.as_o = (float *)(ring + R.stage_o);
  sp.as_lse = (float *)(ring + R.stage_lse);
  sp.match_pos_out = match_pos;
  sp.out = out;
  if (fused) {
    sp.app_pos = (int32_t *)(ring + R.pos);
    sp.app_q = ring + R.q;
    sp.app_o = (float *)(ring + R.o);
    sp.app_lse = (float *)(ring + R.lse);
    sp.as_o = nullptr;
    sp.as_lse = nullptr;
  }
  {
    const bool plain = fused && !t_phase[0] && !t_phase[1] && !t_phase[2];
    sp.early_start = note_launch(sm, ring_ws, plain ? ring_ws : nullptr) && plain ? 1 : 0;
  }
  if (record_phase(0, sm) != cudaSuccess || launch_step(sp, cfg, sm) != cudaSuccess ||
      record_phase(1, sm) != cudaSuccess)
    return MAC_ERR_CUDA;
  if (fused) return record_phase(2, sm) == cudaSuccess ? MAC_OK : MAC_ERR_CUDA;

  AppendParams ap = append_params(cfg, R, ring, sp);
  ap.q_src = ring + R.stage_q;
  if (use_aux) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (cudaEventRecord(ev->main_done, sm) != cudaSuccess ||
        cudaStreamWaitEvent(sa, ev->main_done, 0) != cudaSuccess)
      return MAC_ERR_CUDA;
    if (launch_append(ap, cfg->dtype, sa) != cudaSuccess || record_phase(2, sa) != cudaSuccess)
      return MAC_ERR_CUDA;
    if (cudaEventRecord(ev->aux_done, sa) != cudaSuccess) return MAC_ERR_CUDA;
    ev->pending = true;
    ev->capture_id = cap_id;
  } else {
    if (launch_append(ap, cfg->dtype, sm) != cudaSuccess || record_phase(2, sm) != cudaSuccess)
      return MAC_ERR_CUDA;
  }
  return MAC_OK;
}

int mac_full_attention(const mac_config *cfg, void *scratch_ws, const void *q_pre,
                       const int32_t *seq_len, const mac_kv *kv, float *out, float *lse,
                       void *stream) {
  int v = validate(cfg);
  if (v != MAC_OK) return v;
  if (!scratch_ws || !q_pre || !seq_len || !out || !aligned16(scratch_ws) || !aligned16(q_pre) ||
      !aligned16(out))
    return MAC_ERR_INVALID_ARG;
  if ((v = check_kv(cfg, kv)) != MAC_OK) return v;
  const ScratchLayout S = scratch_layout(cfg);
  StepParams sp = step_params(cfg, S, (uint8_t *)scratch_ws, kv, MODE_FULL);
  sp.pos_base = seq_len;
  sp.q = q_pre;
  sp.out = out;
  sp.out_lse = lse;
  sp.early_start = note_launch((cudaStream_t)stream, nullptr, kNoRing) ? 1 : 0;
  if (launch_step(sp, cfg, (cudaStream_t)stream) != cudaSuccess) return MAC_ERR_CUDA;
  return MAC_OK;
}

int mac_full_attention_noalloc(const mac_config *cfg, const void *q_pre, const int32_t *seq_len,
                               const mac_kv *kv, float *out, float *lse, void *stream) {
  int v = validate(cfg);
  if (v != MAC_OK) return v;
  if (scratch_layout(cfg).total > MAC_NOALLOC_SCRATCH_BYTES) return MAC_ERR_UNSUPPORTED;
  if (!q_pre || !seq_len || !out || !aligned16(q_pre) || !aligned16(out)) return MAC_ERR_INVALID_ARG;
  if ((v = check_kv(cfg, kv)) != MAC_OK) return v;
  void *scratch = noalloc_scratch();
  if (!scratch) return MAC_ERR_CUDA;
  // the previous call left its counters and status in the array: clear the
  // control part (everything before the partials) on this call's stream
  note_launch((cudaStream_t)stream, nullptr, nullptr);  // a memset comes between
  if (cudaMemsetAsync(scratch, 0, scratch_layout(cfg).parts, (cudaStream_t)stream) != cudaSuccess)
    return MAC_ERR_CUDA;
  return mac_full_attention(cfg, scratch, q_pre, seq_len, kv, out, lse, stream);
}

int mac_join_aux(void *ring_ws, void *stream_main) {
  if (!ring_ws) return MAC_ERR_INVALID_ARG;
  cudaStream_t sm = (cudaStream_t)stream_main;
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_rings.find(ring_ws);
  if (it == g_rings.end() || !it->second.pending) return MAC_OK;
  if (it->second.capture_id == capture_id_of(sm)) {
    if (cudaStreamWaitEvent(sm, it->second.aux_done, 0) != cudaSuccess) return MAC_ERR_CUDA;
  }
  it->second.pending = false;
  return MAC_OK;
}

int mac_set_phase_events(void *before_step, void *after_step, void *after_append) {
  t_phase[0] = (cudaEvent_t)before_step;
  t_phase[1] = (cudaEvent_t)after_step;
  t_phase[2] = (cudaEvent_t)after_append;
  return MAC_OK;
}

int mac_set_trace(void *device_buffer) {
  t_trace = (unsigned long long *)device_buffer;
  return MAC_OK;
}

int mac_test_wait_budget(int64_t cycles, int32_t withhold_use) {
  if (cycles < 1 || cycles > kWaitLimit || withhold_use < -1) return MAC_ERR_INVALID_ARG;
  t_wait_limit = cycles;
  t_withhold = withhold_use;
  return MAC_OK;
}

int mac_reset_requests(const mac_config *cfg, void *ring_ws, int32_t *reset_flags, void *stream) {
  int v = validate(cfg);
  if (v != MAC_OK) return v;
  if (!ring_ws || !reset_flags || ((uintptr_t)reset_flags & 3u) != 0) return MAC_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  {
    // after an append still pending on an auxiliary stream for these rings
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_rings.find(ring_ws);
    if (it != g_rings.end() && it->second.pending && it->second.capture_id == capture_id_of(s)) {
      if (cudaStreamWaitEvent(s, it->second.aux_done, 0) != cudaSuccess) return MAC_ERR_CUDA;
    }
  }
  const mac_ring_layout R = ring_layout(cfg);
  int32_t *pos = (int32_t *)((uint8_t *)ring_ws + R.pos);
  note_launch(s, nullptr, nullptr);
  return launch_reset(pos, reset_flags, cfg->batch, cfg->ring_k, s) == cudaSuccess ? MAC_OK : MAC_ERR_CUDA;
}

int mac_release_ring(void *ring_ws) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_rings.find(ring_ws);
  if (it == g_rings.end()) return MAC_OK;
  if (it->second.main_done) cudaEventDestroy(it->second.main_done);
  if (it->second.aux_done) cudaEventDestroy(it->second.aux_done);
  g_rings.erase(it);
  return MAC_OK;
}

int mac_last_status(const mac_config *cfg, void *scratch_ws, int32_t *device_status, void *stream) {
  int v = validate(cfg);
  if (v != MAC_OK) return v;
  if (!scratch_ws || !device_status) return MAC_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  const ScratchLayout S = scratch_layout(cfg);
  int32_t *ctl = (int32_t *)((uint8_t *)scratch_ws + S.ctl);
  int32_t host = 0;
  if (cudaMemcpyAsync(&host, ctl, sizeof host, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess || cudaMemsetAsync(ctl, 0, sizeof host, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return MAC_ERR_CUDA;
  *device_status = host;
  return MAC_OK;
}

}  // extern "C"
