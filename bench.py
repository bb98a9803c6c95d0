#!/usr/bin/env python
"""Benchmark of MAC-Attention decode attention on GB300.

One benchmark step = one decode token through the attention of a stack of
``--layers`` independent layer states (default 32, a Llama-3-8B-deep stack):
for every layer, match -> band+tail/full attention -> rectify-append over the
whole batch.  The default workload is the long-context one: batch 4, 32 query
/ 8 KV heads, d=128, 131072 tokens of context per request, bf16 K/V, ring
K=1024, band r=256, tau=0.6, clustered queries (~99% reuse).

Inputs are synthetic (seeded generators) and resident in HBM before the timed
region; the rings are filled by ring_k untimed decode steps from empty rings,
so the timed steps run at context 131072+1 .. 131072+K with full rings.  The
32 layer states (about 2.2 GB of K/V each) keep every step's working set far
above the 129 MB L2.  A step is one replay of a CUDA graph holding the 32
decode calls; inputs for the step are gathered from the resident arrays by a
device-side step counter.

value = layer-steps/s over all GPUs (1e6 / us per layer step at N=1).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "decode-attention steps/s (us/step) per layer at 32K/128K/256K; HBM GB/s vs peak"
UNIT = "layer-steps/s"
L2_BYTES = 129 * 2 ** 20


# ---------------------------------------------------------------------------
# process group (replicas; the only collectives are a barrier and a max)
# ---------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_group(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def barrier(dist, device=None):
    if dist is not None:
        if device is not None:
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(dist, x: float, device=None) -> float:
    """Max of a scalar over all ranks (the slowest rank defines the time)."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(units_per_rank: float, world: int, t_max: float) -> float:
    """Throughput of the whole job: units all ranks processed / slowest time."""
    return units_per_rank * world / t_max


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = np.array([float(r[1]) for r in rows])
        mx = max(float(r[2]) for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# workload setup
# ---------------------------------------------------------------------------

def run_plan(w, warmup, steps, prof_steps, e2e_steps):
    """Prompt lengths so that the timed steps start right after the target
    context, after ring_k ring-filling steps and the warm-up steps."""
    fill = w.ring_k
    total = fill + warmup + steps + prof_steps + e2e_steps
    prompt = [L - fill - warmup for L in w.contexts]
    return fill, total, w.with_(contexts=prompt, n_steps=total)


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return {}


def ncu_traffic(kernel: str, bytes_per_launch: float):
    """DRAM bytes per launch for this run's mix of launches: the committed
    ncu capture's traffic over the algorithmic bytes of the same launches
    (one layer state, same per-layer workload), times this run's algorithmic
    bytes per launch; None when the kernel's source changed since."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        rec = json.load(open(path))[kernel]
    except (OSError, ValueError, KeyError):
        return None
    src = os.path.join(ROOT, "long_context_decode_gb300", "csrc", rec["source"])
    try:
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    if sha != rec.get("source_sha") or "traffic_over_algorithmic" not in rec:
        return None
    return rec["traffic_over_algorithmic"] * bytes_per_launch


def layer_step_bytes(w, m, mpos, ring_valid, front_sink=0):
    """Algorithmic bytes of one layer step from the match results:
    (match bytes, attend bytes, writes).  m [B]; mpos [B, Hq] (-1 = miss).
    With a front sink F the span starts at F+1 at the earliest and the sink
    [1, min(F, m)] is read besides."""
    B, Hq, Hkv, d, G, r, F = w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim, w.group, w.band_r, front_sink
    from long_context_decode_gb300.workloads import F32
    es = 4 if w.dtype == F32 else 2
    match = sum(Hq * ring_valid[b] * d * es for b in range(B)) + B * Hq * d * es + B * w.ring_k * 4
    attend = 0
    for b in range(B):
        lo = np.where(mpos[b] >= 1, np.maximum(F + 1, mpos[b] - r + 1), F + 1)
        for g in range(Hkv):
            s = int(lo[g * G:(g + 1) * G].min())
            attend += (max(0, int(m[b]) - s + 1) + min(F, int(m[b]))) * 2 * d * es
            if w.page_size:
                attend += ((int(m[b]) - s) // w.page_size + 1) * 4
        attend += int((mpos[b] >= 1).sum()) * (d + 1) * 4
    writes = B * Hq * (d * 4 + d * es + (d + 1) * 4)
    return match, attend, writes


# ---------------------------------------------------------------------------
# the CUDA arm
# ---------------------------------------------------------------------------

# the other contexts the metric names, measured in the same default run
EXTRA_CONTEXTS = ("llama8b-32k", "verylong-256k")


def run_mac(args, rank, world, local):
    import torch

    from long_context_decode_gb300 import build as libbuild
    libbuild.build()

    dist = init_group(world, "nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w0 = select_workload(args)
    out = measure(args, w0, dist, rank, world, dev)
    # 32K and 256K beside the 128K line (one GPU: each is its own replica
    # stack, measured after the main one has released its memory)
    if (world == 1 and args.context_steps > 0 and args.workload == "long-128k" and not args.ring_k
            and not args.front_sink and not args.kv_heads):
        from long_context_decode_gb300.workloads import WORKLOADS
        ctx = {}
        for name in EXTRA_CONTEXTS:
            sub = argparse.Namespace(**vars(args))
            sub.steps, sub.e2e_steps, sub.full_steps, sub.workload = args.context_steps, 0, 2, name
            torch.cuda.empty_cache()
            r = measure(sub, WORKLOADS[name], dist, rank, world, dev)
            ctx[name] = {
                "workload": r["config"]["workload"], "steps": sub.steps, "layers_per_step": sub.layers,
                "us_per_layer_step": r["us_per_layer_step"], "value": r["value"], "unit": UNIT,
                "bytes_per_launch": r["roofline"]["bytes_per_launch"], "launch_us": r["roofline"]["launch_us"],
                "achieved_gbs": r["roofline"]["achieved"], "frac": r["roofline"]["frac"],
                "hit_rate": r["step_roofline"]["hit_rate"], "clocks": r["clocks"],
                "full_attention": r["full_attention"], "device_status": r["device_status"],
            }
        out["contexts"] = ctx
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(w0, args, budget_s=args.cpu_budget)
    return out, rank


def measure(args, w0, dist, rank, world, dev):
    """One workload: the timed decode steps of a stack of layer states, the
    step kernel's roofline, the end-to-end leg and the full-attention leg."""
    import torch

    from long_context_decode_gb300 import mac
    from long_context_decode_gb300.workloads import F32, device_kv, device_paged_kv, device_queries

    Lc, K, Wm, P, E = args.layers, args.steps, args.warmup, args.profile_steps, args.e2e_steps
    fill, total, w = run_plan(w0, Wm, K, P, E)
    B, Hq, Hkv, d = w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim

    # ---- inputs resident in HBM -----------------------------------------
    t_setup = time.time()
    kvs, kv_tensors = [], []
    kv_all = None  # contiguous caches: every layer's K (and V) in one tensor, a layer per slice
    for layer in range(Lc):
        if w.page_size:
            kp, vp, table = device_paged_kv(w.with_(seed=w.seed * 100 + layer), 0, dev)
            tdev = torch.from_numpy(table).to(dev)
            kv_tensors.append((kp, vp, tdev))
            kvs.append(mac.kv_view(kp, vp, tdev))
        else:
            k, v = device_kv(w, w.capacity(), dev, seed_offset=layer)
            if kv_all is None:
                kv_all = (torch.empty((Lc,) + tuple(k.shape), dtype=k.dtype, device=dev),
                          torch.empty((Lc,) + tuple(v.shape), dtype=v.dtype, device=dev))
            kv_all[0][layer].copy_(k)
            kv_all[1][layer].copy_(v)
            del k, v
            kv_tensors.append((kv_all[0][layer], kv_all[1][layer], None))
            kvs.append(mac.kv_view(kv_all[0][layer], kv_all[1][layer]))
    cap = w.capacity() if not w.page_size else kv_tensors[0][2].shape[1] * 16
    q_all = torch.stack([device_queries(w, total, dev, stream_seed=layer).permute(2, 0, 1, 3)
                         for layer in range(Lc)], dim=1).contiguous()  # [total, Lc, B, Hq, d]
    es = 4 if w.dtype == F32 else 2
    cfg = mac.config(B, Hq, Hkv, d, w.ring_k, w.band_r, w.tau, dtype=mac.MAC_F32 if w.dtype == F32 else mac.MAC_BF16,
                     page_size=w.page_size, max_context=cap, front_sink=args.front_sink)
    ring_bytes, scratch_bytes = mac.mac_workspace_size(cfg)
    scratch = torch.zeros(scratch_bytes, dtype=torch.uint8, device=dev)
    layers = [mac.MacLayer(cfg, scratch=scratch, device=dev) for _ in range(Lc)]
    for L in layers:
        mac.mac_init_rings(cfg, L.ring, scratch, None, None, 0, None)
    kv_bytes = sum(t.numel() * t.element_size() for kt in kv_tensors for t in kt[:2])

    q_cur = torch.empty((1, Lc, B, Hq, d), dtype=q_all.dtype, device=dev)
    base = torch.tensor([L + 1 for L in w.contexts], dtype=torch.int64, device=dev)
    seq_cur = torch.empty(B, dtype=torch.int32, device=dev)
    step_ctr = torch.zeros(1, dtype=torch.int64, device=dev)
    outs = torch.empty((Lc, B, Hq, d), dtype=torch.float32, device=dev)
    mpos = torch.empty((Lc, B, Hq), dtype=torch.int32, device=dev)
    main = torch.cuda.Stream(dev)
    # the append: fused into the step kernel (no auxiliary stream), or the
    # append kernel on an auxiliary stream after an event
    aux = torch.cuda.Stream(dev) if args.append == "aux" else None

    def advance(q_src=None):
        if q_src is None:
            torch.index_select(q_all, 0, step_ctr, out=q_cur)
        torch.add(base, step_ctr, out=seq_tmp)
        seq_cur.copy_(seq_tmp)
        step_ctr.add_(1)

    seq_tmp = torch.empty(B, dtype=torch.int64, device=dev)

    def decode_layers(q_src, phase=None):
        for layer in range(Lc):
            if phase is not None:
                mac.mac_set_phase_events(*phase[layer])
            mac.mac_decode_step(cfg, layers[layer].ring, scratch, q_src[layer], seq_cur, kvs[layer],
                                outs[layer], mpos[layer], main, aux)
        for L in layers:
            mac.mac_join_aux(L.ring, main)

    torch.cuda.synchronize(dev)
    g_main = torch.cuda.CUDAGraph()
    with torch.cuda.stream(main):
        with torch.cuda.graph(g_main, stream=main):
            advance()
            decode_layers(q_cur[0])
    # per-kernel timing: the library records these events around its step
    # kernel and after its append, as event-record nodes of the profiled graph
    phase_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(Lc)]
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    for evs in phase_ev:
        for e in evs:
            e.record(main)  # creates the underlying CUDA event
    torch.cuda.synchronize(dev)
    g_prof = torch.cuda.CUDAGraph()
    with torch.cuda.stream(main):
        with torch.cuda.graph(g_prof, stream=main):
            advance()
            decode_layers(q_cur[0], phase=phase_ev)

    # ---- ring fill + warm-up (untimed) ----------------------------------
    with torch.cuda.stream(main):
        for _ in range(fill + Wm):
            g_main.replay()
    torch.cuda.synchronize(dev)
    assert mac.mac_last_status(cfg, scratch) == 0, "device status after warm-up"
    setup_s = time.time() - t_setup

    # ---- timed region ---------------------------------------------------
    clocks = ClockSampler()
    if rank == 0:
        clocks.start()
    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(main):
        t0.record(main)
        for _ in range(K):
            g_main.replay()
        t1.record(main)
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    clk = clocks.stop() if rank == 0 else None
    t_local = t0.elapsed_time(t1) / 1e3
    t_max = max_over_ranks(dist, t_local, dev)
    status = mac.mac_last_status(cfg, scratch)

    # ---- the step's own small kernels, timed alone -----------------------
    # A timed step is the graph: the 4 PyTorch kernels of advance() (query
    # gather, lengths, counter), then the Lc step kernels.  The same 4
    # kernels on dummy outputs (the counter unchanged), replayed alone, give
    # their share; the rest of the timed step, per layer, is the step
    # kernel's time including its launch gap: a duration no longer than the
    # timed layer step.
    ctr_d = torch.zeros(1, dtype=torch.int64, device=dev)
    q_d, seq_tmp_d, seq_d = torch.empty_like(q_cur), torch.empty_like(seq_tmp), torch.empty_like(seq_cur)
    g_adv = torch.cuda.CUDAGraph()
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(main):
        with torch.cuda.graph(g_adv, stream=main):
            torch.index_select(q_all, 0, ctr_d, out=q_d)
            torch.add(base, ctr_d, out=seq_tmp_d)
            seq_d.copy_(seq_tmp_d)
            ctr_d.add_(0)
        g_adv.replay()
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(main)
        for _ in range(200):
            g_adv.replay()
        a1.record(main)
    torch.cuda.synchronize(dev)
    adv_s = a0.elapsed_time(a1) / 1e3 / 200
    launch_s = max(1e-9, (t_max / K - adv_s) / Lc)

    # ---- profiled steps: per-kernel times and algorithmic bytes ----------
    kern_ms, append_ms, step_ms, mb, ab, wb, hits, heads = [], [], [], 0, 0, 0, 0, 0
    for _ in range(P):
        with torch.cuda.stream(main):
            step_ev[0].record(main)
            g_prof.replay()
            step_ev[1].record(main)
        torch.cuda.synchronize(dev)
        step_ms.append(step_ev[0].elapsed_time(step_ev[1]))
        mp = mpos.cpu().numpy()
        m = seq_cur.cpu().numpy().astype(np.int64)
        ring_valid = np.minimum(w.ring_k, m - 1 - (np.array(w.contexts)))
        for layer in range(Lc):
            kern_ms.append(phase_ev[layer][0].elapsed_time(phase_ev[layer][1]))
            append_ms.append(phase_ev[layer][1].elapsed_time(phase_ev[layer][2]))
            a, b_, c = layer_step_bytes(w, m, mp[layer], ring_valid, args.front_sink)
            mb += a
            ab += b_
            wb += c
            hits += int((mp[layer] >= 1).sum())
            heads += mp[layer].size
    n_prof = max(1, P * Lc)
    match_bytes, attend_bytes, write_bytes = mb / n_prof, ab / n_prof, wb / n_prof
    kern_s, append_s = np.mean(kern_ms) / 1e3, np.mean(append_ms) / 1e3
    layer_step_s = np.mean(step_ms) / 1e3 / Lc

    # ---- end to end through host buffers --------------------------------
    e2e = None
    if E > 0 and not w.page_size:
        e2e = run_e2e(torch, mac, cfg, w, layers, scratch, kvs, kv_all, q_all, step_ctr, base,
                      seq_cur, seq_tmp, outs, mpos, main, aux, Lc, E, dev, dist)

    peaks = measured_peaks()
    hbm_peak = peaks.get("hbm_gbs", 6800.0)

    # ---- the miss fallback as its own call: full attention over [1, m] ---
    # (the same layer stack and current lengths; the speedup of the step
    # over it is the method's gain on this workload)
    full = None
    if args.full_steps > 0:
        g_full = torch.cuda.CUDAGraph()
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(main):
            with torch.cuda.graph(g_full, stream=main):
                for layer in range(Lc):
                    mac.mac_full_attention(cfg, scratch, q_cur[0][layer], seq_cur, kvs[layer], outs[layer],
                                           None, main)
            g_full.replay()
            f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            f0.record(main)
            for _ in range(args.full_steps):
                g_full.replay()
            f1.record(main)
        torch.cuda.synchronize(dev)
        full_s = f0.elapsed_time(f1) / 1e3 / (args.full_steps * Lc)
        m_now = seq_cur.cpu().numpy().astype(np.int64)
        full_bytes = float(sum(Hkv * int(m) * 2 * d * es for m in m_now) + B * Hq * d * es)
        full = {"us_per_layer_step": full_s * 1e6, "gbs": full_bytes / full_s / 1e9,
                "frac": full_bytes / full_s / 1e9 / hbm_peak, "bytes_per_layer_step": full_bytes,
                "step_speedup": full_s / (t_max / (K * Lc)), "steps": args.full_steps}
    # the step kernel (match + band/tail attention + merge) is the dominant
    # kernel; the append copies ~1/1000 of its bytes on the aux stream
    dominant = "step_kernel"
    dom_bytes, dom_s = match_bytes + attend_bytes, launch_s
    achieved = dom_bytes / dom_s / 1e9
    us_layer = t_max / (K * Lc) * 1e6
    value = whole_job_value(K * Lc, world, t_max)
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": Wm,
        "ms_per_step": t_max / K * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32" if w.dtype == F32 else "bf16", "data": "synthetic",
        "impl": "mac",
        "config": {
            "workload": f"{w0.name}: {w0.description}",
            "layers_per_step": Lc, "batch": B, "context": w0.contexts[0] if len(set(w0.contexts)) == 1
            else "mixed", "ring_k": w.ring_k, "band_r": w.band_r, "tau": w.tau,
            "threshold": "(1-tau)*sqrt(2d)", "parallelism": f"replicas x{world} (no data-path collective)",
            "l2": f"inputs larger than L2: {Lc} layer states, {kv_bytes / 2**30:.1f} GiB K/V resident, "
                  f"~{(match_bytes + attend_bytes) * Lc / 2**20:.0f} MiB read per step vs 129 MiB L2",
            "rings": f"filled by {fill} untimed decode steps from empty rings",
            "append": ("fused into the step kernel (no auxiliary stream)" if args.append == "fused"
                       else "append kernel on an auxiliary stream after an event"),
            "front_sink": args.front_sink,
        },
        "us_per_layer_step": us_layer,
        # our kernels in the timed region: the step kernel per layer step, plus
        # the append kernel when it runs on the auxiliary stream
        "gpu_launches": (2 if aux is not None else 1) * K * Lc,
        "roofline": {
            "bound": "hbm", "kernel": dominant, "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
            "frac": achieved / hbm_peak, "traffic": ncu_traffic(dominant, dom_bytes),
            "bytes_per_launch": dom_bytes, "launch_us": dom_s * 1e6,
            "launch_us_source": "driver-timed step minus its 4 step-advance kernels (timed alone), per layer",
            "peak_source": "of measured (MEASURED_PEAKS.json hbm_gbs)" if "hbm_gbs" in peaks
            else "of fallback 6.8 TB/s",
        },
        "kernels": {
            "step_kernel": {"us": launch_s * 1e6, "bytes": dom_bytes, "match_bytes": match_bytes,
                            "attend_bytes": attend_bytes, "gbs": dom_bytes / launch_s / 1e9,
                            # the same kernel bracketed by event-record nodes in a second
                            # graph (the nodes themselves add to it)
                            "us_with_event_nodes": kern_s * 1e6},
            "step_advance": {"kernels": 4, "us_per_step": adv_s * 1e6},
            # the ring append: its own kernel after the step on the auxiliary
            # stream, or written by the step kernel's final merges (fused)
            "append": ({"kernel": "append_kernel", "us_after_step": append_s * 1e6, "write_bytes": write_bytes}
                       if aux is not None else {"kernel": "step_kernel (fused)", "write_bytes": write_bytes}),
        },
        "full_attention": full,
        "step_roofline": {
            "algorithmic_read_bytes": match_bytes + attend_bytes, "write_bytes": write_bytes,
            # the whole timed layer step (its share of the step-advance kernels included)
            "us_per_layer_step": us_layer,
            "gbs": (match_bytes + attend_bytes) / (us_layer * 1e-6) / 1e9,
            "frac": (match_bytes + attend_bytes) / (us_layer * 1e-6) / 1e9 / hbm_peak,
            "hit_rate": hits / max(1, heads),
        },
        "clocks": clk,
        "e2e": e2e,
        "device_status": status,
        "setup_s": setup_s,
    }
    for L in layers:
        L.release()
    return out


def run_e2e(torch, mac, cfg, w, layers, scratch, kvs, kv_all, q_all, step_ctr, base, seq_cur,
            seq_tmp, outs, mpos, main, aux, Lc, E, dev, dist):
    """E steps through host buffers: per step, the queries and the new token's
    K/V rows of every layer are copied from pinned host memory (one copy
    each, on a copy stream, into one of two staging sets), the new rows are
    written into every layer's cache (one kernel each for K and V), the
    decode runs, the outputs are copied back, and the host waits for each
    step's result.  Step i+1's copies and launch are queued before the host
    waits for step i, so the copies overlap the previous step's compute."""
    B, Hq, Hkv, d = w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim
    start = int(step_ctr.item())
    k_all, v_all = kv_all
    # host copies of what the next E steps consume
    q_host = q_all[start:start + E].cpu().pin_memory()                 # [E, Lc, B, Hq, d]
    m_steps = [np.array(w.contexts) + 1 + start + i for i in range(E)]
    kv_host = torch.empty((E, 2, B, Lc, Hkv, d), dtype=q_all.dtype).pin_memory()
    bi = torch.arange(B, device=dev)
    for i in range(E):
        idx = torch.from_numpy(m_steps[i] - 1).to(dev)
        kv_host[i, 0] = k_all[:, bi, :, idx].cpu()                     # [B, Lc, Hkv, d]
        kv_host[i, 1] = v_all[:, bi, :, idx].cpu()
    out_h = [torch.empty((Lc, B, Hq, d), dtype=torch.float32).pin_memory() for _ in range(2)]
    out_d = [torch.empty_like(outs) for _ in range(2)]
    q_stage = [torch.empty(q_host.shape[1:], dtype=q_host.dtype, device=dev) for _ in range(2)]
    kv_stage = [torch.empty(kv_host.shape[1:], dtype=kv_host.dtype, device=dev) for _ in range(2)]

    graphs = []
    torch.cuda.synchronize(dev)
    for k in range(2):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(main):
            with torch.cuda.graph(g, stream=main):
                torch.add(base, step_ctr, out=seq_tmp)
                seq_cur.copy_(seq_tmp)
                step_ctr.add_(1)
                rows = seq_tmp - 1
                k_all[:, bi, :, rows] = kv_stage[k][0]
                v_all[:, bi, :, rows] = kv_stage[k][1]
                for layer in range(Lc):
                    mac.mac_decode_step(cfg, layers[layer].ring, scratch, q_stage[k][layer], seq_cur,
                                        kvs[layer], out_d[k][layer], mpos[layer], main, aux)
                for L in layers:
                    mac.mac_join_aux(L.ring, main)
        graphs.append(g)
    copy, back = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    h2d_done = [torch.cuda.Event() for _ in range(2)]
    step_done = [torch.cuda.Event() for _ in range(2)]
    d2h_done = [torch.cuda.Event() for _ in range(2)]

    def launch(i):
        # step i: its inputs into staging set i % 2 once step i-2 is done with
        # it; its replay after those copies (and after step i-2's outputs in
        # set i % 2 were copied back); its outputs back on their own stream
        k = i % 2
        with torch.cuda.stream(copy):
            if i >= 2:
                copy.wait_event(step_done[k])
            q_stage[k].copy_(q_host[i], non_blocking=True)
            kv_stage[k].copy_(kv_host[i], non_blocking=True)
            h2d_done[k].record(copy)
        with torch.cuda.stream(main):
            main.wait_event(h2d_done[k])
            if i >= 2:
                main.wait_event(d2h_done[k])
            graphs[k].replay()
            step_done[k].record(main)
        with torch.cuda.stream(back):
            back.wait_event(step_done[k])
            out_h[k].copy_(out_d[k], non_blocking=True)
            d2h_done[k].record(back)

    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(main):
        t0.record(main)
        launch(0)
        for i in range(E):
            if i + 1 < E:
                launch(i + 1)
            d2h_done[i % 2].synchronize()  # step i's result is on the host
        main.wait_stream(back)
        t1.record(main)
    torch.cuda.synchronize(dev)
    t = max_over_ranks(dist, t0.elapsed_time(t1) / 1e3, dev)
    _, world, _ = dist_env()
    bi_bytes = (q_host[0].numel() + kv_host[0].numel()) * q_host.element_size() + B * 8
    return {"value": whole_job_value(E * Lc, world, t), "unit": UNIT, "steps": E,
            "h2d_bytes_per_step": int(bi_bytes), "d2h_bytes_per_step": int(out_h[0].numel() * 4),
            "path": "pinned host -> device copies of the queries and new K/V rows (copy stream, two staging "
                    "sets), the rows written into every layer's cache, CUDA-graph replay of the layer stack "
                    "through the C ABI, device -> pinned host copy of the outputs, the host waiting for every "
                    "step's result with the next step already queued"}


# ---------------------------------------------------------------------------
# the CPU oracle (baseline / reference arm)
# ---------------------------------------------------------------------------

def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the ISA)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def oracle_sample(w0, warmup, steps, budget_s=None, single_s=0.0):
    """Time the fp64 oracle on request 0 of the workload (all its heads),
    after filling its rings with ring_k untimed decode steps; returns
    (seconds per request-step, steps timed, threads) and, with single_s > 0,
    (seconds per request-step, steps timed) of further steps on one thread
    for about single_s seconds."""
    from long_context_decode_gb300.workloads import F32, host_kv
    from oracle import mac_oracle as O

    fill = w0.ring_k
    wr = w0.with_(batch=1, contexts=[w0.contexts[0] - fill - warmup],
                  n_steps=fill + warmup + steps, page_size=0)
    cap = wr.capacity()
    k, v = host_kv(wr, cap)
    q = wr.query_bits(fill + warmup + steps)
    cfg = O.Config(1, wr.n_q_heads, wr.n_kv_heads, wr.head_dim, wr.ring_k, wr.band_r, wr.tau,
                   dtype=O.F32 if wr.dtype == F32 else O.BF16)
    kv = O.KV(k, v, capacity=cap)
    ring = O.Ring(cfg)
    threads = min(os.cpu_count() or 1, wr.n_q_heads)
    L = wr.contexts[0]
    for s in range(fill + warmup):
        O.decode_step(cfg, ring, np.ascontiguousarray(q[:, :, s]), np.array([L + 1 + s], np.int32),
                      kv, n_threads=threads)
    times = []
    t_start = time.perf_counter()
    # with a one-thread leg, the threaded leg takes at most half the steps
    n_multi = steps // 2 if single_s > 0 else steps
    for s in range(fill + warmup, fill + warmup + n_multi):
        t0 = time.perf_counter()
        O.decode_step(cfg, ring, np.ascontiguousarray(q[:, :, s]), np.array([L + 1 + s], np.int32),
                      kv, n_threads=threads)
        times.append(time.perf_counter() - t0)
        if budget_s is not None and time.perf_counter() - t_start > budget_s:
            break
    if single_s <= 0:
        return float(np.mean(times)), len(times), threads
    one = []
    t_start = time.perf_counter()
    for s in range(fill + warmup + len(times), fill + warmup + steps):
        t0 = time.perf_counter()
        O.decode_step(cfg, ring, np.ascontiguousarray(q[:, :, s]), np.array([L + 1 + s], np.int32),
                      kv, n_threads=1)
        one.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start > single_s:
            break
    return float(np.mean(times)), len(times), threads, (float(np.mean(one)) if one else None), len(one)


def cpu_baseline(w0, args, budget_s=20.0):
    t, n, threads, t1, n1 = oracle_sample(w0, 3, 512, budget_s=budget_s, single_s=budget_s / 2)
    per_layer_step = t * w0.batch  # the oracle sample is one of the batch's requests
    return {"value": 1.0 / per_layer_step, "unit": UNIT, "cores": threads, "kind": "oracle",
            "cpu_model": cpu_model(), "host_cpus": os.cpu_count(),
            "single_thread": ({"value": 1.0 / (t1 * w0.batch), "unit": UNIT, "cores": 1, "steps": n1}
                              if t1 else None),
            "sample": f"fp64 C oracle, request 0 of {w0.batch} (all {w0.n_q_heads} heads, one thread per "
                      f"head up to {threads} threads), {n} decode steps after {w0.ring_k}+3 untimed "
                      f"ring-filling steps at context {w0.contexts[0]}, then {n1} more steps on one thread; "
                      f"time per request-step x {w0.batch} requests = one layer step"}


def select_workload(args):
    """The named workload, with its ring capacity replaced when --ring-k is
    given and its KV-head count when --kv-heads is."""
    from long_context_decode_gb300.workloads import WORKLOADS, with_kv_heads, with_ring_k
    w0 = WORKLOADS[args.workload]
    k = getattr(args, "ring_k", None)
    w0 = with_ring_k(w0, k) if k else w0
    hkv = getattr(args, "kv_heads", None)
    return with_kv_heads(w0, hkv) if hkv else w0


def run_reference(args, rank, world):
    if rank != 0:
        return None, rank
    w0 = select_workload(args)
    t, n, threads = oracle_sample(w0, args.warmup, args.steps)
    per_layer_step = t * w0.batch
    value = 1.0 / per_layer_step
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": n,
        "warmup": args.warmup, "ms_per_step": per_layer_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "impl": "reference",
        "config": {"workload": f"{w0.name}: {w0.description}", "batch": w0.batch,
                   "context": w0.contexts[0], "layers_per_step": 1},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"request 0 of {w0.batch}; per layer step = request-step time x "
                                   f"{w0.batch}"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }, rank


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=8)
    ap.add_argument("--impl", choices=["mac", "reference"], default="mac")
    ap.add_argument("--workload", default="long-128k")
    ap.add_argument("--full-steps", type=int, default=4,
                    help="replays of the full-attention (miss fallback) layer stack timed after the step")
    ap.add_argument("--front-sink", type=int, default=0,
                    help="front-sink isolation: tokens [1, F] out of the summaries, attended every step")
    ap.add_argument("--ring-k", type=int, default=None,
                    help="ring capacity K in place of the workload's (the K sweep, e.g. 512)")
    ap.add_argument("--kv-heads", type=int, default=None,
                    help="KV heads in place of the workload's (another GQA group size; 4 with 32 query heads "
                         "runs the GQA-8 kernel)")
    ap.add_argument("--layers", type=int, default=32)
    ap.add_argument("--profile-steps", type=int, default=8)
    ap.add_argument("--e2e-steps", type=int, default=64)
    ap.add_argument("--cpu-budget", type=float, default=20.0)
    ap.add_argument("--context-steps", type=int, default=1000,
                    help="timed steps of each of the 32K and 256K workloads reported beside the 128K line "
                         "(0: skip them)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--append", choices=["fused", "aux"], default="fused",
                    help="rectify-append inside the step kernel, or as a kernel on an auxiliary stream")
    args = ap.parse_args()
    rank, world, local = dist_env()
    if args.impl == "reference":
        out, rank = run_reference(args, rank, world)
    else:
        out, rank = run_mac(args, rank, world, local)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
