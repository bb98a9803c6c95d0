"""Per-phase profile of the step kernel from its own trace points.

    python -m long_context_decode_gb300.trace [workload] [--layers N] [--reps R]

A stack of ``--layers`` layer states of the workload (its own K/V, rings and
queries each, so a step's working set is far above L2), rings filled by
ring_k untimed decode steps, is replayed from a CUDA graph as in the
benchmark.  In a second graph the last layer's step kernel carries the
phase trace (``mac_set_trace``): per CTA, %globaltimer stamps at the end of
each phase.  Each replay of that graph is one traced step; the table gives,
per phase, the median CTA's and the last CTA's time since the first CTA
started, for steps where every head hits and for steps with one missing
unit.  The traced kernel is a separate instantiation with the stamps
compiled in (the product kernels carry none); a stamp costs a timer read
and a store, so it runs a little slower than the product kernel.

Each class also gets the mean CTA residency (start to end): in a stack of
layers the next kernel's CTAs take each SM as it frees up (early start), so
the SMs stay occupied and the layer step's period is close to this mean.

The stamps follow the span kernel's layout (GQA groups up to 4, bf16
without a front sink; see ``mac_set_trace`` in include/mac.h).
"""
from __future__ import annotations

import argparse
import json
import sys

import numpy as np

# span kernel stamps, in phase order: (index, name)
PHASES = [
    (0, "start"),
    (7, "tail layout published"),
    (8, "first match chunk arrived"),
    (2, "tail pieces done"),
    (1, "match done"),
    (10, "grid barrier passed"),
    (5, "decisions read"),
    (3, "bands laid out"),
    (4, "band pieces and merges done"),
    (6, "end"),
]


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("workload", nargs="?", default="long-128k")
    ap.add_argument("--layers", type=int, default=8)
    ap.add_argument("--reps", type=int, default=48)
    ap.add_argument("--json", default=None, help="also write the per-step rows here")
    args = ap.parse_args(argv)

    import torch

    from . import build as libbuild
    libbuild.build()
    from . import mac
    from .workloads import WORKLOADS, device_kv, device_queries

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w0 = WORKLOADS[args.workload]
    if w0.n_q_heads // w0.n_kv_heads > 4 or w0.page_size:
        sys.exit("the trace table covers the span kernel on contiguous K/V (GQA groups up to 4)")
    NL, R = args.layers, args.reps
    fill, warm = w0.ring_k, 3
    total = fill + warm + 8 + R
    w = w0.with_(contexts=[L - fill - warm for L in w0.contexts], n_steps=total)
    B, Hq, Hkv, d = w.batch, w.n_q_heads, w.n_kv_heads, w.head_dim
    keep, kvs = [], []
    for layer in range(NL):
        k, v = device_kv(w, w.capacity(), dev, seed_offset=layer)
        keep.append((k, v))
        kvs.append(mac.kv_view(k, v))
    q_all = torch.stack([device_queries(w, total, dev, stream_seed=layer).permute(2, 0, 1, 3)
                         for layer in range(NL)], 1).contiguous()
    cfg = mac.config(B, Hq, Hkv, d, w.ring_k, w.band_r, w.tau, max_context=w.capacity())
    scratch = torch.zeros(mac.mac_workspace_size(cfg)[1], dtype=torch.uint8, device=dev)
    layers = [mac.MacLayer(cfg, scratch=scratch, device=dev) for _ in range(NL)]
    for L in layers:
        mac.mac_init_rings(cfg, L.ring, scratch, None, None, 0, None)
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    TP = 32
    base = torch.tensor([c + 1 for c in w.contexts], dtype=torch.int64, device=dev)
    ctr = torch.zeros(1, dtype=torch.int64, device=dev)
    seq = torch.empty(B, dtype=torch.int32, device=dev)
    qcur = torch.empty((1, NL, B, Hq, d), dtype=q_all.dtype, device=dev)
    out = torch.empty(NL, B, Hq, d, device=dev)
    mps = torch.empty(NL, B, Hq, dtype=torch.int32, device=dev)
    trace = torch.zeros(nsm * TP, dtype=torch.int64, device=dev)
    main_s = torch.cuda.Stream(dev)

    def body(traced):
        torch.index_select(q_all, 0, ctr, out=qcur)
        seq.copy_((base + ctr).to(torch.int32))
        ctr.add_(1)
        for layer in range(NL):
            if traced and layer == NL - 1:
                mac.mac_set_trace(trace)
            mac.mac_decode_step(cfg, layers[layer].ring, scratch, qcur[0, layer], seq, kvs[layer], out[layer],
                                mps[layer], main_s, None)

    graphs = {}
    torch.cuda.synchronize()
    for traced in (False, True):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(main_s):
            with torch.cuda.graph(g, stream=main_s):
                body(traced)
        graphs[traced] = g
    with torch.cuda.stream(main_s):
        for _ in range(fill + warm):
            graphs[False].replay()
    torch.cuda.synchronize()
    rows = []
    for _ in range(R):
        trace.zero_()
        with torch.cuda.stream(main_s):
            graphs[True].replay()
        torch.cuda.synchronize()
        t = trace.view(nsm, TP).cpu().numpy().astype(np.int64)
        miss = mps[NL - 1].cpu().numpy().reshape(B, Hkv, Hq // Hkv) < 0
        t0 = t[:, 0][t[:, 0] != 0].min()
        row = {"missing_heads": int(miss.sum()), "missing_units": int(miss.any(-1).sum())}
        for k, name in PHASES:
            col = t[:, k]
            col = col[col != 0]
            if len(col):
                c = (col - t0) / 1e3
                row[name] = (float(np.median(c)), float(c.max()))
        # CTA residency: start to end of each CTA, averaged over the CTAs.  In
        # a stack of layers the next kernel's CTAs take each SM as it frees
        # up, so the layer step's period is close to this mean.
        ran = (t[:, 0] != 0) & (t[:, 6] != 0)
        row["residency_us"] = float(np.mean((t[ran, 6] - t[ran, 0]) / 1e3)) if ran.any() else None
        clk = (t[:, 17] - t[:, 16]) / np.maximum(1, t[:, 6] - t[:, 0])
        row["sm_ghz"] = float(np.median(clk[clk > 0])) if (clk > 0).any() else None
        # per-CTA band work: the last band piece's tiles done (stamp 24, us),
        # time waiting for band tiles (25, ns), band tokens (22) and pieces
        # (23), time merging (18, ns) and units merged (19)
        has = t[:, 24] != 0
        if has.any():
            row["band_tiles_done_us"] = [float(np.percentile((t[has, 24] - t0) / 1e3, q)) for q in (10, 50, 90, 100)]
        row["band_wait_us"] = [float(np.percentile(t[:, 25] / 1e3, q)) for q in (50, 90, 100)]
        row["band_tokens"] = [float(np.percentile(t[:, 22], q)) for q in (10, 50, 90, 100)]
        row["band_pieces"] = [float(np.percentile(t[:, 23], q)) for q in (50, 100)]
        row["merge_us"] = [float(np.percentile(t[:, 18] / 1e3, q)) for q in (50, 90, 100)]
        row["units_merged"] = [float(np.percentile(t[:, 19], q)) for q in (50, 100)]
        row["longest_merge_us"] = float(t[:, 20].max() / 1e3)
        row["longest_merge_entries"] = int(t[np.argmax(t[:, 20]), 21])
        rows.append(row)
    status = mac.mac_last_status(cfg, scratch)

    def table(sel):
        if not sel:
            return None
        return {name: (float(np.median([r[name][0] for r in sel if name in r])),
                       float(np.median([r[name][1] for r in sel if name in r])))
                for _, name in PHASES if any(name in r for r in sel)}

    hit = [r for r in rows if r["missing_units"] == 0]
    miss1 = [r for r in rows if r["missing_units"] == 1]
    t_hit, t_miss = table(hit), table(miss1)
    print(f"# step kernel phases: {w0.name}, last of {NL} layer states, {R} traced steps "
          f"({len(hit)} all-hit, {len(miss1)} with one missing unit); device status {status}")
    print()
    print("| phase (stamp) | all hit: median CTA | all hit: last CTA | one missing unit: median CTA | "
          "one missing unit: last CTA |")
    print("|---|---|---|---|---|")
    for k, name in PHASES:
        a = t_hit.get(name) if t_hit else None
        b = t_miss.get(name) if t_miss else None
        fa = (f"{a[0]:.2f}", f"{a[1]:.2f}") if a else ("-", "-")
        fb = (f"{b[0]:.2f}", f"{b[1]:.2f}") if b else ("-", "-")
        print(f"| {name} ({k}) | {fa[0]} | {fa[1]} | {fb[0]} | {fb[1]} |")
    for label, sel in (("all hit", hit), ("one missing unit", miss1)):
        if not sel:
            continue
        print()
        print(f"{label}, per-CTA band work (medians over the steps of percentiles over the CTAs):")
        for key in ("band_tiles_done_us", "band_wait_us", "band_tokens", "band_pieces", "merge_us", "units_merged"):
            vals = [r[key] for r in sel if key in r]
            if vals:
                print(f"  {key}: " + " / ".join(f"{v:.2f}" for v in np.median(np.array(vals), 0)))
        print(f"  longest merge: {np.median([r['longest_merge_us'] for r in sel]):.2f} us, "
              f"{int(np.median([r['longest_merge_entries'] for r in sel]))} entries")
        res = [r["residency_us"] for r in sel if r["residency_us"] is not None]
        if res:
            print(f"  CTA residency (start to end, mean over the CTAs): {np.median(res):.2f} us")
    ghz = [r["sm_ghz"] for r in rows if r["sm_ghz"]]
    print()
    print(f"µs since the first CTA started; medians over the steps of each class. SM clock during the "
          f"traced kernels: {np.median(ghz):.2f} GHz." if ghz else "")
    if args.json:
        json.dump(rows, open(args.json, "w"))
    for L in layers:
        L.release()


if __name__ == "__main__":
    main()
