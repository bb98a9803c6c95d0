"""Seeded synthetic inputs for MAC-Attention decode steps.

This module only draws data: query processes, K/V values, page tables and
the workload shapes.  It holds none of the method's arithmetic, imports
neither the CUDA binding nor the oracle, and is the one module both sides'
tests and the benchmark share.

The pages evaluate on LongBench v2, RULER and LongGenBench with real models;
none of those are available, so these generators stand in for them with the
shapes of the workloads the benchmark names and query processes tuned to the
hit rates those workloads are described with (clustered queries for a ~99%
reuse rate, AR(1) with random jumps for mixed hits and misses).

Position convention: positions are 1-based, the prompt has L tokens, and
decode step s (0-based) runs at length m = L + 1 + s with the K/V of
position m already in the cache.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

BF16, F32 = 0, 1


# --------------------------------------------------------------------------
# bf16 bit patterns
# --------------------------------------------------------------------------

def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even) and
    return the 16-bit patterns as uint16."""
    f = np.ascontiguousarray(x, np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    nan = np.isnan(f)
    out = rounded.astype(np.uint16)
    out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.ascontiguousarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# query processes (per head, independent)
# --------------------------------------------------------------------------

def ar1_queries(rng: np.random.Generator, n_heads: int, n_pos: int, d: int, rho: float,
                sigma: float, jump_prob=0.0) -> np.ndarray:
    """q_1 ~ N(0, I); q_t = rho q_{t-1} + sigma eps, and with probability
    ``jump_prob`` (scalar or one value per head) a fresh q_t ~ N(0, I).
    Returns [n_heads, n_pos, d] float32."""
    jp = np.broadcast_to(np.asarray(jump_prob, np.float64), (n_heads,))
    q = np.empty((n_heads, n_pos, d), np.float32)
    cur = rng.standard_normal((n_heads, d))
    q[:, 0] = cur
    for t in range(1, n_pos):
        eps = rng.standard_normal((n_heads, d))
        nxt = rho * cur + sigma * eps
        jump = rng.random(n_heads) < jp
        if jump.any():
            nxt[jump] = rng.standard_normal((int(jump.sum()), d))
        cur = nxt
        q[:, t] = cur
    return q


def clustered_queries(rng: np.random.Generator, n_heads: int, n_pos: int, d: int,
                      n_centroids: int = 16, sigma: float = 0.05,
                      switch_prob: float = 0.01) -> np.ndarray:
    """Per head: n_centroids centroids ~ N(0, I); q_t = c_{z_t} + sigma eps,
    where z switches to a uniformly drawn centroid with probability
    ``switch_prob`` per position.  Returns [n_heads, n_pos, d] float32."""
    cent = rng.standard_normal((n_heads, n_centroids, d))
    z = np.empty((n_heads, n_pos), np.int64)
    z[:, 0] = rng.integers(0, n_centroids, n_heads)
    for t in range(1, n_pos):
        sw = rng.random(n_heads) < switch_prob
        z[:, t] = np.where(sw, rng.integers(0, n_centroids, n_heads), z[:, t - 1])
    heads = np.arange(n_heads)[:, None]
    q = cent[heads, z] + sigma * rng.standard_normal((n_heads, n_pos, d))
    return q.astype(np.float32)


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------

@dataclass
class Workload:
    """Shape, parameters and generators of one synthetic decode workload."""
    name: str
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    contexts: list            # prompt length L per request
    ring_k: int
    band_r: int
    tau: float
    dtype: int                # BF16 or F32 for queries and K/V
    page_size: int            # 0 = contiguous cache
    n_steps: int
    seed: int
    query: str                # "ar1_jump", "clustered", "ar1_098", "ar1_skew"
    keys: str                 # "normal", "heavy_hitters", "recency"
    description: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)

    # ---- queries --------------------------------------------------------
    def queries(self, n_pos: int, seed_offset: int = 0) -> np.ndarray:
        """[B, Hq, n_pos, d] pre-RoPE queries (float32, already rounded to
        the workload dtype's precision)."""
        rng = np.random.default_rng([self.seed, 1, seed_offset])
        H = self.batch * self.n_q_heads
        d = self.head_dim
        if self.query == "ar1_jump":
            q = ar1_queries(rng, H, n_pos, d, 0.95, 0.31, 1.0 / 8.0)
        elif self.query == "clustered":
            q = clustered_queries(rng, H, n_pos, d, 16, 0.05, 0.01)
        elif self.query == "ar1_098":
            q = ar1_queries(rng, H, n_pos, d, 0.98, float(np.sqrt(1 - 0.98 ** 2)), 0.0)
        elif self.query == "ar1_skew":
            per_group = np.array([0.1, 0.3, 0.5, 0.7])
            jp = np.tile(per_group[np.arange(self.n_q_heads) % self.group % 4], self.batch)
            q = ar1_queries(rng, H, n_pos, d, 0.95, 0.31, jp)
        else:
            raise ValueError(self.query)
        q = q.reshape(self.batch, self.n_q_heads, n_pos, d)
        return q

    def query_bits(self, n_pos: int, seed_offset: int = 0) -> np.ndarray:
        """Queries as the raw buffer the library and the oracle read."""
        q = self.queries(n_pos, seed_offset)
        return to_bf16_bits(q) if self.dtype == BF16 else np.ascontiguousarray(q, np.float32)

    # ---- keys / values --------------------------------------------------
    def key_scale(self, b: int, positions: np.ndarray) -> np.ndarray:
        """Per-position key scale (1 except for the structured key sets)."""
        L = self.contexts[b]
        if self.keys == "recency":
            # key norm decays with distance from the end of the prompt
            # (decode positions keep the largest scale)
            dist = np.maximum(L - positions, 0)
            return 0.25 + 1.75 * np.exp(-dist / 4096.0)
        return np.ones(positions.shape, np.float64)

    def heavy_hitters(self, b: int) -> np.ndarray:
        """[Hkv, 4] heavy-hitter positions (1-based) of request b, uniform in
        [1, L]; their keys are scaled x4."""
        rng = np.random.default_rng([self.seed, 2, b])
        return rng.integers(1, self.contexts[b] + 1, size=(self.n_kv_heads, 4))

    def capacity(self, extra_steps: int = 0) -> int:
        """Tokens of cache each request needs for the prompt plus the
        decode steps (rounded up to the page size)."""
        need = max(self.contexts) + self.n_steps + extra_steps
        ps = self.page_size or 16
        return (need + ps - 1) // ps * ps


# The five workloads the benchmark configuration names.  Seeds: 0 for the
# tiny case (as given), 1-4 for the others.
WORKLOADS = {
    "tiny-4k": Workload(
        "tiny-4k", 1, 1, 1, 128, [4096], 64, 32, 0.6, F32, 0, 64, 0, "ar1_jump", "normal",
        "batch 1, 1 q/1 kv head, d=128, context 4096, K=64, r=32, tau=0.6, fp32 Q/K/V; "
        "AR(1) 0.95/0.31 queries with 1-in-8 jumps; 64 steps"),
    "llama8b-32k": Workload(
        "llama8b-32k", 1, 32, 8, 128, [32768], 1024, 256, 0.6, BF16, 0, 256, 1, "clustered",
        "heavy_hitters",
        "Llama-3-8B-like layer: batch 1, 32q/8kv, d=128, context 32768, bf16 K/V with 4 heavy "
        "hitters x4, K=1024, r=256, tau=0.6, clustered queries; 256 steps"),
    "long-128k": Workload(
        "long-128k", 4, 32, 8, 128, [131072] * 4, 1024, 256, 0.6, BF16, 0, 256, 2, "clustered",
        "heavy_hitters",
        "batch 4, 32q/8kv, d=128, context 131072 per request, bf16 KV, K=1024, r=256, "
        "tau=0.6, clustered queries (~99% hit); 256 steps"),
    "verylong-256k": Workload(
        "verylong-256k", 1, 32, 8, 128, [262144], 1024, 256, 0.75, BF16, 0, 128, 3, "ar1_098",
        "recency",
        "batch 1, 32q/8kv, d=128, context 262144, bf16 KV, K=1024, r=256, tau=0.75; AR(1) "
        "rho=0.98 queries, recency-biased key norms; 128 steps"),
    "mixed-paged": Workload(
        "mixed-paged", 16, 32, 8, 128,
        [int(x) for x in np.random.default_rng([4, 0]).integers(8192, 131072 + 1, 16)],
        1024, 256, 0.45, BF16, 16, 128, 4, "ar1_skew", "normal",
        "16 requests, contexts U[8K,128K], 32q/8kv, d=128, bf16 KV in 16-token pages with a "
        "shuffled page table, K=1024, r=256, tau=0.45; AR(1) queries with per-head jump "
        "probabilities 0.1/0.3/0.5/0.7 inside each GQA group (~60% hit); 128 steps"),
}


def with_ring_k(w: Workload, ring_k: int) -> Workload:
    """The same workload with another ring capacity K (the ring-size sweep)."""
    if ring_k == w.ring_k:
        return w
    return w.with_(ring_k=ring_k, name=f"{w.name}-k{ring_k}",
                   description=w.description.replace(f"K={w.ring_k}", f"K={ring_k}"))


def with_kv_heads(w: Workload, n_kv_heads: int) -> Workload:
    """The same workload with another number of KV heads (another GQA group
    size: 32q/4kv runs the GQA-8 path)."""
    if n_kv_heads == w.n_kv_heads:
        return w
    if n_kv_heads < 1 or w.n_q_heads % n_kv_heads:
        raise ValueError(f"{n_kv_heads} KV heads do not divide {w.n_q_heads} query heads")
    return w.with_(n_kv_heads=n_kv_heads, name=f"{w.name}-kv{n_kv_heads}",
                   description=w.description.replace(f"{w.n_q_heads}q/{w.n_kv_heads}kv",
                                                     f"{w.n_q_heads}q/{n_kv_heads}kv"))


def shuffled_page_table(rng: np.random.Generator, batch: int, pages_per_req: int) -> np.ndarray:
    """[B, pages_per_req] physical page ids: a random permutation of all pages."""
    perm = rng.permutation(batch * pages_per_req).astype(np.int32)
    return perm.reshape(batch, pages_per_req)


# --------------------------------------------------------------------------
# host-side K/V (small cases; large caches are drawn on the device)
# --------------------------------------------------------------------------

def host_kv(w: Workload, capacity: int, seed_offset: int = 0):
    """Contiguous K, V [B, Hkv, capacity, d] as raw buffers (uint16 bf16
    patterns or float32), with the workload's key structure applied."""
    rng = np.random.default_rng([w.seed, 3, seed_offset])
    shape = (w.batch, w.n_kv_heads, capacity, w.head_dim)
    k = rng.standard_normal(shape, dtype=np.float32)
    v = rng.standard_normal(shape, dtype=np.float32)
    pos = np.arange(1, capacity + 1)
    for b in range(w.batch):
        k[b] *= w.key_scale(b, pos)[None, :, None].astype(np.float32)
        if w.keys == "heavy_hitters":
            hh = w.heavy_hitters(b)
            for g in range(w.n_kv_heads):
                k[b, g, hh[g] - 1] *= 4.0
    if w.dtype == BF16:
        return to_bf16_bits(k), to_bf16_bits(v)
    return k, v


def paginate(k: np.ndarray, v: np.ndarray, page_size: int, rng: np.random.Generator):
    """Scatter contiguous [B, Hkv, cap, d] caches into shuffled pages
    [n_pages, Hkv, page_size, d]; returns (k_pages, v_pages, page_table)."""
    B, H, cap, d = k.shape
    assert cap % page_size == 0
    ppr = cap // page_size
    table = shuffled_page_table(rng, B, ppr)
    kp = np.empty((B * ppr, H, page_size, d), k.dtype)
    vp = np.empty_like(kp)
    for b in range(B):
        kb = k[b].reshape(H, ppr, page_size, d).transpose(1, 0, 2, 3)
        vb = v[b].reshape(H, ppr, page_size, d).transpose(1, 0, 2, 3)
        kp[table[b]] = kb
        vp[table[b]] = vb
    return kp, vp, table


# --------------------------------------------------------------------------
# device-side K/V (large caches: drawn on the GPU with a seeded generator)
# --------------------------------------------------------------------------

def device_kv(w: Workload, capacity: int, device, seed_offset: int = 0):
    """Contiguous K, V [B, Hkv, capacity, d] drawn on ``device`` (torch
    generator seeded from the workload), key structure applied, stored in the
    workload dtype (torch.bfloat16 or torch.float32)."""
    import torch

    gen = torch.Generator(device=device)
    gen.manual_seed(int(w.seed) * 1000 + 17 + seed_offset)
    shape = (w.batch, w.n_kv_heads, capacity, w.head_dim)
    dt = torch.bfloat16 if w.dtype == BF16 else torch.float32
    k = torch.empty(shape, dtype=dt, device=device)
    v = torch.empty(shape, dtype=dt, device=device)
    pos = np.arange(1, capacity + 1)
    for b in range(w.batch):
        for g in range(w.n_kv_heads):
            kb = torch.randn((capacity, w.head_dim), generator=gen, device=device)
            vb = torch.randn((capacity, w.head_dim), generator=gen, device=device)
            if w.keys == "recency":
                sc = torch.from_numpy(w.key_scale(b, pos).astype(np.float32)).to(device)
                kb *= sc[:, None]
            if w.keys == "heavy_hitters":
                hh = torch.from_numpy(w.heavy_hitters(b)[g] - 1).to(device)
                kb[hh] *= 4.0
            k[b, g] = kb.to(dt)
            v[b, g] = vb.to(dt)
    return k, v


def device_queries(w: Workload, n_pos: int, device, stream_seed: int = 0):
    """[B, Hq, n_pos, d] pre-RoPE queries drawn on ``device`` with the
    workload's query process (same processes as ``Workload.queries``, drawn
    with a torch generator), stored in the workload dtype."""
    import torch

    gen = torch.Generator(device=device)
    gen.manual_seed(int(w.seed) * 7919 + 101 + int(stream_seed))
    H, d = w.batch * w.n_q_heads, w.head_dim
    f32 = dict(device=device, dtype=torch.float32)
    if w.query == "clustered":
        cent = torch.randn((H, 16, d), generator=gen, **f32)
        switch = torch.rand((H, n_pos), generator=gen, **f32) < 0.01
        switch[:, 0] = True
        newz = torch.randint(0, 16, (H, n_pos), generator=gen, device=device)
        t = torch.arange(n_pos, device=device).expand(H, n_pos)
        last = torch.cummax(torch.where(switch, t, torch.zeros_like(t)), dim=1).values
        z = newz.gather(1, last)
        q = cent[torch.arange(H, device=device)[:, None], z]
        q += 0.05 * torch.randn((H, n_pos, d), generator=gen, **f32)
    else:
        if w.query == "ar1_jump":
            rho, sigma, jp = 0.95, 0.31, torch.full((H,), 1.0 / 8.0, **f32)
        elif w.query == "ar1_098":
            rho, sigma, jp = 0.98, float(np.sqrt(1 - 0.98 ** 2)), torch.zeros((H,), **f32)
        elif w.query == "ar1_skew":
            per = torch.tensor([0.1, 0.3, 0.5, 0.7], **f32)
            jp = per[torch.arange(w.n_q_heads, device=device) % w.group % 4].repeat(w.batch)
            rho, sigma = 0.95, 0.31
        else:
            raise ValueError(w.query)
        q = torch.empty((H, n_pos, d), **f32)
        cur = torch.randn((H, d), generator=gen, **f32)
        q[:, 0] = cur
        for i in range(1, n_pos):
            nxt = rho * cur + sigma * torch.randn((H, d), generator=gen, **f32)
            jump = torch.rand((H,), generator=gen, **f32) < jp
            cur = torch.where(jump[:, None], torch.randn((H, d), generator=gen, **f32), nxt)
            q[:, i] = cur
    dt = torch.bfloat16 if w.dtype == BF16 else torch.float32
    return q.view(w.batch, w.n_q_heads, n_pos, d).to(dt)


def device_paged_kv(w: Workload, extra_steps: int, device, page_seed: int = 5):
    """Paged K, V [n_pages, Hkv, 16, d] on ``device`` holding each request's
    own ceil((L_b + steps)/16) pages at shuffled physical ids, and the page
    table [B, max_pages] (int32, -1 past a request's last page)."""
    import torch

    ps = 16
    need = [(L + w.n_steps + extra_steps + ps - 1) // ps for L in w.contexts]
    total, max_pages = sum(need), max(need)
    perm = np.random.default_rng([page_seed, w.seed]).permutation(total).astype(np.int32)
    table = np.full((w.batch, max_pages), -1, np.int32)
    off = 0
    for b, n in enumerate(need):
        table[b, :n] = perm[off:off + n]
        off += n
    gen = torch.Generator(device=device)
    gen.manual_seed(int(w.seed) * 1000 + 29)
    dt = torch.bfloat16 if w.dtype == BF16 else torch.float32
    shape = (total, w.n_kv_heads, ps, w.head_dim)
    kp = torch.empty(shape, dtype=dt, device=device)
    vp = torch.empty(shape, dtype=dt, device=device)
    for b, n in enumerate(need):
        ids = torch.from_numpy(table[b, :n].astype(np.int64)).to(device)
        for g in range(w.n_kv_heads):
            kb = torch.randn((n * ps, w.head_dim), generator=gen, device=device)
            vb = torch.randn((n * ps, w.head_dim), generator=gen, device=device)
            if w.keys == "heavy_hitters":
                kb[torch.from_numpy(w.heavy_hitters(b)[g] - 1).to(device)] *= 4.0
            kp[ids, g] = kb.view(n, ps, w.head_dim).to(dt)
            vp[ids, g] = vb.view(n, ps, w.head_dim).to(dt)
    return kp, vp, table
