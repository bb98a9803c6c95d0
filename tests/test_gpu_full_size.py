"""Parity at the benchmark workloads' full sizes (32K, 4 x 128K, 256K, 16
mixed paged requests of 8K-128K), with the kernels' production launch
configuration: trajectories from empty rings, every (request, head)
decision compared every step, outputs compared on a seeded sample of heads
(the oracle computes those heads' attention; the match runs for all)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from harness import TOL, Problem, compare, gpu_trajectory, oracle_trajectory  # noqa: E402
from long_context_decode_gb300 import mac  # noqa: E402
from long_context_decode_gb300.workloads import WORKLOADS, with_ring_k  # noqa: E402
from oracle import mac_oracle as O  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_decode_gb300 import build as b
    b.build()
    mac.load()


@pytest.mark.parametrize("name,steps,sample,ring_k,sink", [
    ("llama8b-32k", 40, 12, None, 0),
    ("long-128k", 24, 12, None, 0),
    ("long-128k", 24, 12, 512, 0),  # the ring-size sweep's K = 512
    ("long-128k", 16, 8, None, 128),  # front-sink isolation, F = 128
    ("verylong-256k", 24, 8, None, 0),
    ("mixed-paged", 12, 12, None, 0),
    ("gqa8-128k", 16, 8, None, 0),  # 32 q / 4 kv heads (GQA 8) at 2 x 128K
])
def test_full_size_workload(name, steps, sample, ring_k, sink):
    if name == "gqa8-128k":
        w = WORKLOADS["long-128k"].with_(batch=2, contexts=[131072, 100000], n_kv_heads=4, n_steps=steps)
    else:
        w = WORKLOADS[name].with_(n_steps=steps)
    if ring_k:
        w = with_ring_k(w, ring_k)
    P = Problem(w, device_generated=True, native_paged=w.page_size > 0)
    rng = np.random.default_rng(123)
    mask = np.zeros((w.batch, w.n_q_heads), np.uint8)
    flat = rng.choice(w.batch * w.n_q_heads, size=min(sample, w.batch * w.n_q_heads), replace=False)
    mask.reshape(-1)[flat] = 1
    gpu, st, layer = gpu_trajectory(P, steps, cfg=P.cfg(front_sink=sink))
    ref = oracle_trajectory(P, steps, head_mask=mask, front_sink=sink)
    c = compare(gpu, ref, O.threshold_sq(128, w.tau), head_mask=mask)
    assert st == 0
    assert c["mismatched"] == 0, c
    assert c["max_err"] <= TOL, c
    assert c["hits"] > 0
    layer.release()


@pytest.mark.parametrize("query,tau,rope", [
    ("clustered", 0.6, mac.MAC_ROPE_HALF),
    ("ar1_skew", 0.45, mac.MAC_ROPE_HALF),
    ("clustered", 0.6, mac.MAC_ROPE_INTERLEAVED),
])
def test_full_rings_several_match_chunks(query, tau, rope):
    # The ring state the benchmark times: K = 1024 valid candidates per head
    # from the first step on (seeded rings), i.e. 8 match chunks of 128 rows
    # per head dealt to 8 different CTAs whose minima meet in one atomic
    # per head; chunks whose ring positions start past slot 0; decode steps
    # overwriting the oldest slots (wraparound).  Batch, heads, K and r of the
    # 4 x 128K workload at shorter, ragged contexts, so the oracle can seed
    # the sampled heads' summaries.  Every decision every step; outputs of the
    # sampled heads.
    w = WORKLOADS["long-128k"].with_(contexts=[6000, 9001, 12345, 7777], n_steps=40, query=query,
                                     tau=tau)
    P = Problem(w, n_seed=w.ring_k, device_generated=True)
    rng = np.random.default_rng(7)
    mask = np.zeros((w.batch, w.n_q_heads), np.uint8)
    mask.reshape(-1)[rng.choice(w.batch * w.n_q_heads, size=12, replace=False)] = 1
    orope = {mac.MAC_ROPE_HALF: O.ROPE_HALF, mac.MAC_ROPE_INTERLEAVED: O.ROPE_INTERLEAVED}[rope]
    gpu, st, layer = gpu_trajectory(P, w.n_steps, cfg=P.cfg(rope_mode=rope))
    ref = oracle_trajectory(P, w.n_steps, head_mask=mask, rope_mode=orope)
    c = compare(gpu, ref, O.threshold_sq(128, w.tau), head_mask=mask)
    assert st == 0
    assert c["mismatched"] == 0, c
    assert c["max_err"] <= TOL, c
    assert c["hits"] > 0
    # clustered queries match back across the whole ring (several chunks
    # per head); AR(1) queries match the most recent positions
    far = sum(int(((r["match_pos"] >= 1) & (P.m(s)[:, None] - r["match_pos"] > 128)).sum())
              for s, r in enumerate(ref))
    assert far > 0 or query != "clustered"
    layer.release()
