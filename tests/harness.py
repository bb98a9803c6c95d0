"""Helpers shared by the GPU parity tests: build one synthetic problem, run
it through the C ABI and through the fp64 oracle on the same raw inputs, and
compare.  Decisions must match exactly except where the oracle flags them
(minimum within 1e-6 of the threshold, or a runner-up within 1e-6 of the
minimum); outputs must agree to max_i |o - o_ref| / max_i |o_ref| <= 2e-3
per (request, head)."""
from __future__ import annotations

import numpy as np
import torch

from long_context_decode_gb300 import mac
from long_context_decode_gb300.workloads import (BF16, F32, Workload, device_kv, device_paged_kv,
                                                 host_kv, paginate)
from oracle import mac_oracle as O

TOL = 2e-3


def to_dev(a: np.ndarray, dev):
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(a).to(dev)


def to_host_raw(t: torch.Tensor) -> np.ndarray:
    t = t.contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def rel_err(got: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Per (b, h): max_i |got - ref| / max_i |ref|."""
    den = np.abs(ref).max(-1)
    return np.abs(got - ref).max(-1) / np.where(den > 0, den, 1.0)


class Problem:
    """Workload shapes + inputs on host and device."""

    def __init__(self, w: Workload, n_seed: int = 0, paged: bool = False, dev="cuda",
                 device_generated: bool = False, extra: int = 0, page_seed: int = 5,
                 native_paged: bool = False):
        self.w, self.n_seed, self.paged, self.dev = w, n_seed, paged, torch.device(dev)
        self.native_paged = native_paged
        self.cap = w.capacity(extra)
        self.L = np.array(w.contexts, np.int32)
        self.q = w.query_bits(n_seed + w.n_steps + extra)  # positions L-n_seed+1 ...
        if native_paged:
            # each request holds only its own pages (no padding to the longest)
            self.paged = True
            self.kp_dev, self.vp_dev, self.table = device_paged_kv(w, extra, self.dev, page_seed)
            self.table_dev = torch.from_numpy(self.table).to(self.dev)
            self.kp, self.vp = to_host_raw(self.kp_dev), to_host_raw(self.vp_dev)
            self.cap = self.table.shape[1] * 16
            return
        if device_generated:
            self.k_dev, self.v_dev = device_kv(w, self.cap, self.dev)
            self.k, self.v = to_host_raw(self.k_dev), to_host_raw(self.v_dev)
        else:
            self.k, self.v = host_kv(w, self.cap)
            self.k_dev, self.v_dev = to_dev(self.k, self.dev), to_dev(self.v, self.dev)
        if paged:
            kp, vp, table = paginate(self.k, self.v, 16, np.random.default_rng(page_seed))
            self.kp_dev, self.vp_dev = to_dev(kp, self.dev), to_dev(vp, self.dev)
            self.table_dev = torch.from_numpy(table).to(self.dev)

    def cfg(self, **kw) -> mac.mac_config:
        w = self.w
        base = dict(head_dim=w.head_dim, ring_k=w.ring_k, band_r=w.band_r, tau=w.tau,
                    dtype=mac.MAC_F32 if w.dtype == F32 else mac.MAC_BF16,
                    page_size=16 if self.paged else 0, max_context=self.cap)
        base.update(kw)
        return mac.config(w.batch, w.n_q_heads, w.n_kv_heads, **base)

    def ocfg(self, **kw) -> O.Config:
        w = self.w
        base = dict(head_dim=w.head_dim, ring_k=w.ring_k, band_r=w.band_r, tau=w.tau,
                    dtype=O.F32 if w.dtype == F32 else O.BF16,
                    page_size=16 if self.native_paged else 0)
        base.update(kw)
        return O.Config(w.batch, w.n_q_heads, w.n_kv_heads, **base)

    def kv(self) -> mac.mac_kv:
        if self.paged:
            return mac.kv_view(self.kp_dev, self.vp_dev, self.table_dev)
        return mac.kv_view(self.k_dev, self.v_dev)

    def okv(self) -> O.KV:
        if self.native_paged:
            return O.KV(self.kp, self.vp, self.table, max_pages=self.table.shape[1])
        return O.KV(self.k, self.v, capacity=self.cap)

    def q_step(self, s: int) -> np.ndarray:
        return np.ascontiguousarray(self.q[:, :, self.n_seed + s])

    def q_seed(self) -> np.ndarray:
        return np.ascontiguousarray(self.q[:, :, :self.n_seed])

    def m(self, s: int) -> np.ndarray:
        return (self.L + 1 + s).astype(np.int32)


def gpu_trajectory(P: Problem, steps: int, cfg=None, aux=False, graph=False, layer=None):
    """Run `steps` decode steps through the C ABI; returns [(out, match_pos)]."""
    cfg = cfg or P.cfg()
    layer = layer or mac.MacLayer(cfg, device=P.dev)
    kv = P.kv()
    if P.n_seed:
        mac.mac_init_rings(cfg, layer.ring, layer.scratch, to_dev(P.q_seed(), P.dev),
                           torch.from_numpy(P.L).to(P.dev), P.n_seed, kv)
    else:
        mac.mac_init_rings(cfg, layer.ring, layer.scratch, None, None, 0, None)
    B, H, d = P.w.batch, P.w.n_q_heads, P.w.head_dim
    qs = [to_dev(P.q_step(s), P.dev) for s in range(steps)]
    ms = [torch.from_numpy(P.m(s)).to(P.dev) for s in range(steps)]
    outs = [torch.empty(B, H, d, device=P.dev) for _ in range(steps)]
    mps = [torch.empty(B, H, dtype=torch.int32, device=P.dev) for _ in range(steps)]
    main = torch.cuda.current_stream(P.dev)
    side = torch.cuda.Stream(P.dev) if aux else None
    torch.cuda.synchronize(P.dev)

    def run():
        for s in range(steps):
            mac.mac_decode_step(cfg, layer.ring, layer.scratch, qs[s], ms[s], kv, outs[s], mps[s],
                                main, side)
        if aux:
            mac.mac_join_aux(layer.ring, main)

    if graph:
        g = torch.cuda.CUDAGraph()
        cap_stream = torch.cuda.Stream(P.dev)
        with torch.cuda.stream(cap_stream):
            main = cap_stream
            with torch.cuda.graph(g, stream=cap_stream):
                run()
        g.replay()
    else:
        run()
    torch.cuda.synchronize(P.dev)
    status = mac.mac_last_status(cfg, layer.scratch)
    res = [(o.double().cpu().numpy(), p.cpu().numpy()) for o, p in zip(outs, mps)]
    return res, status, layer


def oracle_trajectory(P: Problem, steps: int, head_mask=None, **cfg_kw):
    ocfg = P.ocfg(**cfg_kw)
    ring = O.Ring(ocfg)
    okv = P.okv()
    if P.n_seed:
        O.seed_rings(ocfg, ring, P.q_seed(), P.L, okv, head_mask=head_mask)
    return [O.decode_step(ocfg, ring, P.q_step(s), P.m(s), okv, head_mask=head_mask)
            for s in range(steps)]


# Largest share of decisions the oracle may flag (and the comparison then
# skip): near-ties and distances at the threshold are rare on these inputs,
# so a larger share means the comparison is no longer testing decisions.
MAX_FLAGGED = 0.01


def compare(gpu, ref, thr2, head_mask=None, tol=TOL):
    """Returns dict(decisions, flagged, mismatched, max_err, hits); raises if
    more than MAX_FLAGGED of the decisions (at least 2) were flagged."""
    n = fl = bad = hits = 0
    max_err = 0.0
    for (out, mp), r in zip(gpu, ref):
        f = O.flags(r, thr2)
        ok = ~f
        n += int(ok.sum())
        fl += int(f.sum())
        bad += int((mp[ok] != r["match_pos"][ok]).sum())
        hits += int((r["match_pos"] >= 1).sum())
        mask = np.ones(mp.shape, bool) if head_mask is None else head_mask.astype(bool)
        e = rel_err(out, r["out"])[mask]
        if e.size:
            max_err = max(max_err, float(e.max()))
    assert fl <= max(2, MAX_FLAGGED * (n + fl)), f"{fl} of {n + fl} decisions flagged"
    return dict(decisions=n, flagged=fl, mismatched=bad, max_err=max_err, hits=hits)
