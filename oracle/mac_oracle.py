"""ctypes front end of the fp64 CPU oracle (``mac_oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference arm may import this module; the product
path never does.  It imports nothing from the CUDA package and shares no code
with it.  Inputs are the same raw buffers the CUDA path reads (bf16 bit
patterns as ``uint16`` or ``float32``), converted to fp64 inside the C code.

What each function computes, and the passage it follows, is documented in
``mac_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "mac_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
DEFAULT_LIB = os.path.join(BUILD_DIR, "libmac_oracle.so")

BF16, F32 = 0, 1
THR_ONE_MINUS_TAU, THR_TAU = 0, 1
ROPE_HALF, ROPE_INTERLEAVED, ROPE_NONE = 0, 1, 2


class OcConfig(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int), ("n_q_heads", ctypes.c_int),
        ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
        ("ring_k", ctypes.c_int), ("band_r", ctypes.c_int),
        ("tau", ctypes.c_double), ("thr_mode", ctypes.c_int),
        ("rope_base", ctypes.c_double), ("rope_mode", ctypes.c_int),
        ("dtype", ctypes.c_int), ("page_size", ctypes.c_int),
        ("min_context", ctypes.c_int), ("front_sink", ctypes.c_int),
    ]


class OcKv(ctypes.Structure):
    _fields_ = [
        ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("page_table", ctypes.c_void_p), ("capacity", ctypes.c_int64),
        ("max_pages", ctypes.c_int32),
    ]


class OcRing(ctypes.Structure):
    _fields_ = [
        ("pos", ctypes.c_void_p), ("q", ctypes.c_void_p), ("sM", ctypes.c_void_p),
        ("sZ", ctypes.c_void_p), ("sS", ctypes.c_void_p),
    ]


def build(src: str = SRC, out: str = DEFAULT_LIB, force: bool = False) -> str:
    """Compile the oracle with gcc (portable flags; no FMA contraction so the
    same source gives the same fp64 rounding on x86 and Arm)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                    "-o", tmp, src, "-lm", "-lpthread"], check=True)
    os.replace(tmp, out)
    return out


_LIB = None


def lib() -> ctypes.CDLL:
    """Load the oracle library (``MAC_ORACLE_LIB`` overrides the path)."""
    global _LIB
    if _LIB is None:
        path = os.environ.get("MAC_ORACLE_LIB") or build()
        L = ctypes.CDLL(path)
        vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        L.oc_threshold_sq.argtypes = [i32, dbl, i32]
        L.oc_threshold_sq.restype = dbl
        L.oc_rope.argtypes = [vp, i64, i32, dbl, i32, vp]
        L.oc_summary.argtypes = [vp, vp, i32, i32, vp, i64, i64, vp, vp, vp]
        L.oc_merge.argtypes = [i32, vp, vp, vp, dbl, dbl, vp]
        L.oc_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32]
        L.oc_decode_step.restype = i32
        L.oc_full_attention.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32]
        L.oc_full_attention.restype = i32
        L.oc_seed_rings.argtypes = [vp, vp, vp, vp, i32, vp, vp, i32]
        L.oc_reset_requests.argtypes = [vp, vp, vp]
        L.oc_seed_rings.restype = i32
        _LIB = L
    return _LIB


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


@dataclass
class Config:
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int = 128
    ring_k: int = 1024
    band_r: int = 256
    tau: float = 0.6
    thr_mode: int = THR_ONE_MINUS_TAU
    rope_base: float = 10000.0
    rope_mode: int = ROPE_HALF
    dtype: int = BF16
    page_size: int = 0
    min_context: int = 0
    front_sink: int = 0  # F: [1, F] kept out of the summaries, attended exactly every step

    def c(self) -> OcConfig:
        return OcConfig(self.batch, self.n_q_heads, self.n_kv_heads, self.head_dim,
                        self.ring_k, self.band_r, float(self.tau), self.thr_mode,
                        float(self.rope_base), self.rope_mode, self.dtype, self.page_size,
                        self.min_context, self.front_sink)


@dataclass
class KV:
    """K/V as the CUDA path reads them: contiguous [B, Hkv, capacity, d] or
    paged [n_pages, Hkv, page_size, d] plus a page table [B, max_pages]."""
    k: np.ndarray
    v: np.ndarray
    page_table: np.ndarray | None = None
    capacity: int = 0
    max_pages: int = 0
    _keep: list = field(default_factory=list)

    def c(self) -> OcKv:
        k = np.ascontiguousarray(self.k)
        v = np.ascontiguousarray(self.v)
        pt = None if self.page_table is None else np.ascontiguousarray(self.page_table, np.int32)
        self._keep = [k, v, pt]
        return OcKv(k.ctypes.data, v.ctypes.data, None if pt is None else pt.ctypes.data,
                    int(self.capacity), int(self.max_pages))


class Ring:
    """fp64 ring state: positions [B, K], queries [B, Hq, K, d], summaries."""

    def __init__(self, cfg: Config):
        B, H, K, d = cfg.batch, cfg.n_q_heads, cfg.ring_k, cfg.head_dim
        self.pos = np.zeros((B, K), np.int32)
        self.q = np.zeros((B, H, K, d), np.float64)
        self.sM = np.full((B, H, K), -np.inf)
        self.sZ = np.zeros((B, H, K))
        self.sS = np.zeros((B, H, K, d))

    def c(self) -> OcRing:
        return OcRing(_ptr(self.pos), _ptr(self.q), _ptr(self.sM), _ptr(self.sZ), _ptr(self.sS))

    def copy(self) -> "Ring":
        r = Ring.__new__(Ring)
        for n in ("pos", "q", "sM", "sZ", "sS"):
            setattr(r, n, getattr(self, n).copy())
        return r


def _raw(x: np.ndarray, dtype: int) -> np.ndarray:
    want = np.uint16 if dtype == BF16 else np.float32
    if x.dtype != want:
        raise TypeError(f"expected {want} input, got {x.dtype}")
    return np.ascontiguousarray(x)


def _threads(n: int | None) -> int:
    return n if n else (os.cpu_count() or 1)


def threshold_sq(head_dim: int, tau: float, thr_mode: int = THR_ONE_MINUS_TAU) -> float:
    return lib().oc_threshold_sq(head_dim, float(tau), thr_mode)


def rope(x: np.ndarray, pos: int, base: float = 10000.0, mode: int = ROPE_HALF) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float64)
    out = np.empty_like(x)
    lib().oc_rope(_ptr(x), int(pos), x.shape[-1], float(base), mode, _ptr(out))
    return out


def summary(cfg: Config, kv: KV, b: int, g: int, q_rot: np.ndarray, lo: int, hi: int):
    """(M, Z, S) of rotated query q_rot over tokens [lo, hi] of (b, g)."""
    q = np.ascontiguousarray(q_rot, np.float64)
    M, Z = ctypes.c_double(), ctypes.c_double()
    S = np.zeros(cfg.head_dim)
    c, k = cfg.c(), kv.c()
    lib().oc_summary(ctypes.byref(c), ctypes.byref(k), b, g, _ptr(q), lo, hi,
                     ctypes.byref(M), ctypes.byref(Z), _ptr(S))
    return M.value, Z.value, S


def merge(a, x):
    """(M, Z, S) (+) (M, Z, S)."""
    M, Z = ctypes.c_double(a[0]), ctypes.c_double(a[1])
    S = np.array(a[2], np.float64, copy=True)
    xs = np.ascontiguousarray(x[2], np.float64)
    lib().oc_merge(S.shape[0], ctypes.byref(M), ctypes.byref(Z), _ptr(S), float(x[0]),
                   float(x[1]), _ptr(xs))
    return M.value, Z.value, S


def decode_step(cfg: Config, ring: Ring, q_pre: np.ndarray, seq_len: np.ndarray, kv: KV,
                head_mask: np.ndarray | None = None, n_threads: int | None = None) -> dict:
    """One decode step; mutates ``ring`` (append).  Returns out [B, Hq, d],
    match_pos [B, Hq] (-1 = miss), dmin and dsecond [B, Hq]."""
    B, H, d = cfg.batch, cfg.n_q_heads, cfg.head_dim
    q = _raw(q_pre, cfg.dtype)
    sl = np.ascontiguousarray(seq_len, np.int32)
    hm = None if head_mask is None else np.ascontiguousarray(head_mask, np.uint8)
    out = np.zeros((B, H, d))
    mp = np.zeros((B, H), np.int32)
    dmin = np.zeros((B, H))
    dsec = np.zeros((B, H))
    c, k, rc = cfg.c(), kv.c(), ring.c()
    rcode = lib().oc_decode_step(ctypes.byref(c), ctypes.byref(rc), _ptr(q), _ptr(sl),
                                 ctypes.byref(k), _ptr(hm), _ptr(out), _ptr(mp), _ptr(dmin),
                                 _ptr(dsec), _threads(n_threads))
    if rcode != 0:
        raise ValueError(f"oc_decode_step returned {rcode}")
    return {"out": out, "match_pos": mp, "dmin": dmin, "dsecond": dsec}


def full_attention(cfg: Config, q_pre: np.ndarray, seq_len: np.ndarray, kv: KV,
                   head_mask: np.ndarray | None = None, n_threads: int | None = None):
    """Exact attention over [1, m]: (out [B, Hq, d], lse [B, Hq])."""
    B, H, d = cfg.batch, cfg.n_q_heads, cfg.head_dim
    q = _raw(q_pre, cfg.dtype)
    sl = np.ascontiguousarray(seq_len, np.int32)
    hm = None if head_mask is None else np.ascontiguousarray(head_mask, np.uint8)
    out = np.zeros((B, H, d))
    lse = np.zeros((B, H))
    c, k = cfg.c(), kv.c()
    rcode = lib().oc_full_attention(ctypes.byref(c), _ptr(q), _ptr(sl), ctypes.byref(k),
                                    _ptr(hm), _ptr(out), _ptr(lse), _threads(n_threads))
    if rcode != 0:
        raise ValueError(f"oc_full_attention returned {rcode}")
    return out, lse


def seed_rings(cfg: Config, ring: Ring, q_seed: np.ndarray, prompt_len: np.ndarray, kv: KV,
               head_mask: np.ndarray | None = None, n_threads: int | None = None) -> None:
    """Seed the last n_seed prompt positions with exact summaries."""
    q = _raw(q_seed, cfg.dtype)
    n_seed = q.shape[2]
    pl = np.ascontiguousarray(prompt_len, np.int32)
    hm = None if head_mask is None else np.ascontiguousarray(head_mask, np.uint8)
    c, k, rc = cfg.c(), kv.c(), ring.c()
    rcode = lib().oc_seed_rings(ctypes.byref(c), ctypes.byref(rc), _ptr(q), _ptr(pl), n_seed,
                                ctypes.byref(k), _ptr(hm), _threads(n_threads))
    if rcode != 0:
        raise ValueError(f"oc_seed_rings returned {rcode}")


def reset_requests(cfg: Config, ring: Ring, flags_b: np.ndarray) -> None:
    """Requests whose flag is non-zero start over with an empty ring."""
    f = np.ascontiguousarray(flags_b, np.int32)
    assert f.shape == (cfg.batch,)
    c, rc = cfg.c(), ring.c()
    rcode = lib().oc_reset_requests(ctypes.byref(c), ctypes.byref(rc), _ptr(f))
    if rcode != 0:
        raise ValueError(f"oc_reset_requests returned {rcode}")


def flags(res: dict, thr2: float, rel: float = 1e-6) -> np.ndarray:
    """Decisions excluded from the bit-exact count: minimum distance within
    ``rel`` of the threshold, or a runner-up within ``rel`` of the minimum."""
    dmin, dsec = res["dmin"], res["dsecond"]
    fin = np.isfinite(dmin)
    both = fin & np.isfinite(dsec)
    near_thr = fin & (np.abs(np.where(fin, dmin, 0.0) - thr2) <= rel * thr2)
    gap = np.where(both, dsec, 0.0) - np.where(both, dmin, 0.0)
    near_tie = both & (gap <= rel * np.where(both, dmin, 0.0))
    return near_thr | near_tie
