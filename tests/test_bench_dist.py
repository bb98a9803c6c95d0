"""The benchmark's multi-rank host logic on CPU: world_size-2 gloo process
groups stand in for the per-GPU ranks (one process per GPU, replicas with no
data-path collective; the only collectives are the timing barrier and the
max over ranks)."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, times, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, w, local = bench.dist_env()
    dist = bench.init_group(w, "gloo")
    bench.barrier(dist)
    t_max = bench.max_over_ranks(dist, times[rank])
    value = bench.whole_job_value(1000.0, w, t_max)
    bench.barrier(dist)
    q.put((r, w, local, t_max, value))
    dist.destroy_process_group()


def _run(world, times):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=180) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return out


def test_two_ranks_take_the_slowest_time_and_the_whole_job_units():
    # rank 1 is slower: both ranks report its time, and the job's throughput
    # counts the units of both ranks over it
    out = _run(2, [0.5, 2.0])
    assert [o[0] for o in out] == [0, 1]
    assert all(o[1] == 2 for o in out)
    assert [o[2] for o in out] == [0, 1]
    assert all(o[3] == 2.0 for o in out)
    assert all(o[4] == pytest.approx(1000.0 * 2 / 2.0) for o in out)


def test_single_rank_has_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.init_group(1, "gloo") is None
    assert bench.max_over_ranks(None, 3.5) == 3.5
    bench.barrier(None)
    assert bench.whole_job_value(10.0, 1, 2.0) == 5.0


def test_reference_arm_runs_on_rank_zero_only():
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        workload, steps, warmup = "tiny", 1, 0

    out, rank = bench.run_reference(Args, 1, 2)
    assert out is None and rank == 1


def test_layer_step_bytes_counts_band_tail_and_sink():
    # the algorithmic-bytes model: a miss reads [1, m]; a hit at p reads
    # [p-r+1, m] plus its cached summary; a front sink F starts every span at
    # F+1 and adds the sink [1, min(F, m)]
    sys.path.insert(0, ROOT)
    import numpy as np
    import bench
    from long_context_decode_gb300.workloads import WORKLOADS
    w = WORKLOADS["llama8b-32k"].with_(batch=1)
    d, G, r, Hkv, Hq = w.head_dim, w.group, w.band_r, w.n_kv_heads, w.n_q_heads
    m = np.array([10000])
    row = 2 * d * 2  # K and V bytes per token
    miss = np.full((1, Hq), -1)
    hit = np.full((1, Hq), 9000)
    _, a_miss, _ = bench.layer_step_bytes(w, m, miss, np.array([w.ring_k]))
    _, a_hit, _ = bench.layer_step_bytes(w, m, hit, np.array([w.ring_k]))
    assert a_miss == Hkv * 10000 * row
    assert a_hit == Hkv * (10000 - (9000 - r + 1) + 1) * row + Hq * (d + 1) * 4
    F = 128
    _, s_miss, _ = bench.layer_step_bytes(w, m, miss, np.array([w.ring_k]), F)
    _, s_hit, _ = bench.layer_step_bytes(w, m, hit, np.array([w.ring_k]), F)
    assert s_miss == a_miss  # [F+1, m] and [1, F]: the same tokens
    assert s_hit == a_hit + Hkv * F * row
    # a context inside the sink: everything is sink
    _, s_small, _ = bench.layer_step_bytes(w, np.array([100]), miss, np.array([0]), F)
    assert s_small == Hkv * 100 * row
