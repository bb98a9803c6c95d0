"""Thin ctypes binding of libmac_gb300.so (the C ABI in include/mac.h).

The functions keep the C names and only marshal arguments: every step of
the decode path runs in the library's CUDA kernels.  PyTorch provides the
device memory and streams (``MacLayer`` allocates the workspaces).  There is
no fallback: loading fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

MAC_OK, MAC_ERR_INVALID_ARG, MAC_ERR_UNSUPPORTED, MAC_ERR_CUDA = 0, -1, -2, -3
MAC_DEV_BAD_SEQ_LEN, MAC_DEV_BAD_PAGE, MAC_DEV_WAIT_TIMEOUT, MAC_DEV_NONFINITE_Q, MAC_DEV_BAD_COPY = 1, 2, 4, 8, 16
MAC_TRACE_POINTS = 32
MAC_BF16, MAC_F32 = 0, 1
MAC_THR_ONE_MINUS_TAU, MAC_THR_TAU = 0, 1
MAC_ROPE_HALF, MAC_ROPE_INTERLEAVED, MAC_ROPE_NONE = 0, 1, 2

# every function the header declares (checked against include/mac.h by the tests)
EXPORTS = ("mac_workspace_size", "mac_ring_layout_of", "mac_init_rings", "mac_decode_step",
           "mac_full_attention", "mac_full_attention_noalloc", "mac_join_aux", "mac_release_ring",
           "mac_last_status", "mac_set_phase_events", "mac_set_trace", "mac_status_string",
           "mac_threshold_sq", "mac_reset_requests", "mac_test_wait_budget")
MAC_NOALLOC_SCRATCH_BYTES = 16 << 20


class mac_config(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("ring_k", ctypes.c_int32), ("band_r", ctypes.c_int32),
        ("tau", ctypes.c_double), ("thr_mode", ctypes.c_int32), ("rope_base", ctypes.c_double),
        ("rope_mode", ctypes.c_int32), ("dtype", ctypes.c_int32), ("page_size", ctypes.c_int32),
        ("min_context", ctypes.c_int32), ("max_context", ctypes.c_int64),
        ("front_sink", ctypes.c_int32),
    ]


class mac_kv(ctypes.Structure):
    _fields_ = [
        ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("page_table", ctypes.c_void_p),
        ("capacity", ctypes.c_int64), ("max_pages", ctypes.c_int32), ("n_pages", ctypes.c_int32),
    ]


class mac_ring_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("pos", "q", "o", "lse", "stage_q", "stage_o", "stage_lse", "ctl", "total")]


class MacError(RuntimeError):
    pass


_LIB = None


def lib_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libmac_gb300.so (raises if it has not been built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = lib_path()
    if not os.path.exists(path):
        raise MacError(f"{path} is missing: build it with long_context_decode_gb300.build.build()")
    L = ctypes.CDLL(path)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    P = ctypes.POINTER
    L.mac_workspace_size.argtypes = [P(mac_config), P(ctypes.c_size_t), P(ctypes.c_size_t)]
    L.mac_ring_layout_of.argtypes = [P(mac_config), P(mac_ring_layout)]
    L.mac_init_rings.argtypes = [P(mac_config), vp, vp, vp, vp, i32, P(mac_kv), vp]
    L.mac_decode_step.argtypes = [P(mac_config), vp, vp, vp, vp, P(mac_kv), vp, vp, vp, vp]
    L.mac_full_attention.argtypes = [P(mac_config), vp, vp, vp, P(mac_kv), vp, vp, vp]
    L.mac_full_attention_noalloc.argtypes = [P(mac_config), vp, vp, P(mac_kv), vp, vp, vp]
    L.mac_join_aux.argtypes = [vp, vp]
    L.mac_release_ring.argtypes = [vp]
    L.mac_last_status.argtypes = [P(mac_config), vp, P(i32), vp]
    L.mac_set_phase_events.argtypes = [vp, vp, vp]
    L.mac_set_trace.argtypes = [vp]
    L.mac_reset_requests.argtypes = [P(mac_config), vp, vp, vp]
    L.mac_test_wait_budget.argtypes = [i64, i32]
    L.mac_status_string.argtypes = [ctypes.c_int]
    L.mac_status_string.restype = ctypes.c_char_p
    L.mac_threshold_sq.argtypes = [P(mac_config)]
    L.mac_threshold_sq.restype = ctypes.c_float
    for n in EXPORTS:
        if n not in ("mac_status_string", "mac_threshold_sq"):
            getattr(L, n).restype = ctypes.c_int
    _LIB = L
    return L


def _check(code: int, what: str) -> None:
    if code != MAC_OK:
        raise MacError(f"{what}: {load().mac_status_string(code).decode()} ({code})")


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


# ---------------------------------------------------------------------------
# the C entry points, same names, marshalling only
# ---------------------------------------------------------------------------

def mac_workspace_size(cfg: mac_config) -> tuple[int, int]:
    ring, scratch = ctypes.c_size_t(), ctypes.c_size_t()
    _check(load().mac_workspace_size(ctypes.byref(cfg), ctypes.byref(ring), ctypes.byref(scratch)),
           "mac_workspace_size")
    return ring.value, scratch.value


def mac_ring_layout_of(cfg: mac_config) -> mac_ring_layout:
    lay = mac_ring_layout()
    _check(load().mac_ring_layout_of(ctypes.byref(cfg), ctypes.byref(lay)), "mac_ring_layout_of")
    return lay


def mac_init_rings(cfg, ring, scratch, q_seed, prompt_len, n_seed, kv: mac_kv, stream=None):
    _check(load().mac_init_rings(ctypes.byref(cfg), _ptr(ring), _ptr(scratch), _ptr(q_seed),
                                 _ptr(prompt_len), int(n_seed),
                                 ctypes.byref(kv) if kv is not None else None, _stream(stream)),
           "mac_init_rings")


def mac_decode_step(cfg, ring, scratch, q_pre, seq_len, kv: mac_kv, out, match_pos=None,
                    stream_main=None, stream_aux=None):
    _check(load().mac_decode_step(ctypes.byref(cfg), _ptr(ring), _ptr(scratch), _ptr(q_pre),
                                  _ptr(seq_len), ctypes.byref(kv), _ptr(out), _ptr(match_pos),
                                  _stream(stream_main), _stream(stream_aux)), "mac_decode_step")


def mac_full_attention(cfg, scratch, q_pre, seq_len, kv: mac_kv, out, lse=None, stream=None):
    _check(load().mac_full_attention(ctypes.byref(cfg), _ptr(scratch), _ptr(q_pre), _ptr(seq_len),
                                     ctypes.byref(kv), _ptr(out), _ptr(lse), _stream(stream)),
           "mac_full_attention")


def mac_full_attention_noalloc(cfg, q_pre, seq_len, kv: mac_kv, out, lse=None, stream=None):
    """mac_full_attention with its scratch in the library's fixed array
    (for callers that cannot allocate device memory; see include/mac.h)."""
    _check(load().mac_full_attention_noalloc(ctypes.byref(cfg), _ptr(q_pre), _ptr(seq_len),
                                             ctypes.byref(kv), _ptr(out), _ptr(lse), _stream(stream)),
           "mac_full_attention_noalloc")


def mac_join_aux(ring, stream_main=None):
    _check(load().mac_join_aux(_ptr(ring), _stream(stream_main)), "mac_join_aux")


def mac_release_ring(ring):
    _check(load().mac_release_ring(_ptr(ring)), "mac_release_ring")


def mac_last_status(cfg, scratch, stream=None) -> int:
    st = ctypes.c_int32()
    _check(load().mac_last_status(ctypes.byref(cfg), _ptr(scratch), ctypes.byref(st), _stream(stream)),
           "mac_last_status")
    return st.value


def mac_set_phase_events(before_match=None, after_match=None, after_attend=None):
    """Arm the next mac_decode_step on this thread to record these
    torch.cuda.Event objects (or raw cudaEvent_t handles)."""
    def h(e):
        if e is None or isinstance(e, int):
            return e
        return e.cuda_event
    _check(load().mac_set_phase_events(h(before_match), h(after_match), h(after_attend)),
           "mac_set_phase_events")


def mac_set_trace(buffer):
    """Arm the next step kernel on this thread to write per-CTA phase
    timestamps into ``buffer`` (a torch uint64/int64 tensor of >= 8 * SMs)."""
    _check(load().mac_set_trace(_ptr(buffer)), "mac_set_trace")


def mac_reset_requests(cfg: mac_config, ring, reset_flags, stream=None):
    """Requests whose flag (device int32 tensor [B]) is set start over with
    empty rings: their next step misses on every head; the flags are
    cleared on the device."""
    _check(load().mac_reset_requests(ctypes.byref(cfg), _ptr(ring), _ptr(reset_flags), _stream(stream)),
           "mac_reset_requests")


def mac_test_wait_budget(cycles: int, withhold_use: int = -1):
    """Test hook: the next step kernel on this thread gives every bounded
    wait ``cycles`` SM cycles and never copies stage use ``withhold_use``."""
    _check(load().mac_test_wait_budget(int(cycles), int(withhold_use)), "mac_test_wait_budget")


def mac_status_string(code: int) -> str:
    return load().mac_status_string(code).decode()


def mac_threshold_sq(cfg: mac_config) -> float:
    return float(load().mac_threshold_sq(ctypes.byref(cfg)))


# ---------------------------------------------------------------------------
# convenience: configuration and torch-allocated workspaces
# ---------------------------------------------------------------------------

def config(batch, n_q_heads, n_kv_heads, head_dim=128, ring_k=1024, band_r=256, tau=0.6,
           thr_mode=MAC_THR_ONE_MINUS_TAU, rope_base=10000.0, rope_mode=MAC_ROPE_HALF,
           dtype=MAC_BF16, page_size=0, min_context=0, max_context=131072, front_sink=0) -> mac_config:
    return mac_config(batch, n_q_heads, n_kv_heads, head_dim, ring_k, band_r, float(tau), thr_mode,
                      float(rope_base), rope_mode, dtype, page_size, min_context, int(max_context),
                      int(front_sink))


def kv_view(k, v, page_table=None, capacity=0, max_pages=0, n_pages=0) -> mac_kv:
    """K/V descriptor from torch tensors (contiguous [B, Hkv, cap, d] or
    paged [n_pages, Hkv, 16, d] + page table [B, max_pages])."""
    if page_table is None:
        capacity = capacity or k.shape[2]
    else:
        max_pages = max_pages or page_table.shape[1]
        n_pages = n_pages or k.shape[0]
    return mac_kv(_ptr(k), _ptr(v), _ptr(page_table), int(capacity), int(max_pages), int(n_pages))


class MacLayer:
    """One layer's ring workspace plus a (possibly shared) scratch workspace,
    allocated with torch on the current CUDA device."""

    def __init__(self, cfg: mac_config, scratch=None, device="cuda"):
        import torch
        self.cfg = cfg
        ring_bytes, scratch_bytes = mac_workspace_size(cfg)
        self.ring = torch.zeros(ring_bytes, dtype=torch.uint8, device=device)
        self.scratch = scratch if scratch is not None else torch.zeros(scratch_bytes, dtype=torch.uint8,
                                                                        device=device)
        self.layout = mac_ring_layout_of(cfg)

    def ring_view(self, part: str):
        """A typed torch view of one part of the ring workspace."""
        import torch
        c, L = self.cfg, self.layout
        B, H, K, d = c.batch, c.n_q_heads, c.ring_k, c.head_dim
        qdt = torch.bfloat16 if c.dtype == MAC_BF16 else torch.float32
        spec = {
            "pos": (L.pos, torch.int32, (B, K)),
            "q": (L.q, qdt, (B, H, K, d)),
            "o": (L.o, torch.float32, (B, H, K, d)),
            "lse": (L.lse, torch.float32, (B, H, K)),
            "stage_q": (L.stage_q, qdt, (B, H, d)),
            "stage_o": (L.stage_o, torch.float32, (B, H, d)),
            "stage_lse": (L.stage_lse, torch.float32, (B, H)),
        }[part]
        off, dt, shape = spec
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.empty((), dtype=dt).element_size()
        return self.ring[off:off + nbytes].view(dt).view(shape)

    def release(self):
        mac_release_ring(self.ring)
