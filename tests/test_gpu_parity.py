"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the
same seeded inputs, plus the bitwise self-consistency properties the design
promises (a miss equals full attention, paged equals contiguous, runs are
deterministic, aux-stream and graph-captured runs equal eager ones)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from harness import TOL, Problem, compare, gpu_trajectory, oracle_trajectory, rel_err, to_dev  # noqa: E402
from long_context_decode_gb300 import mac  # noqa: E402
from long_context_decode_gb300.workloads import BF16, F32, WORKLOADS, Workload  # noqa: E402
from oracle import mac_oracle as O  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_decode_gb300 import build as b
    b.build()
    mac.load()


def W(name="t", B=2, Hq=8, Hkv=2, ctx=(700, 1500), K=64, r=32, tau=0.6, dtype=BF16, steps=8,
      seed=11, query="ar1_jump", keys="normal"):
    return Workload(name, B, Hq, Hkv, 128, list(ctx), K, r, tau, dtype, 0, steps, seed, query, keys)


def full_attention_gpu(P, cfg, lens):
    B, H = P.w.batch, P.w.n_q_heads
    q = to_dev(P.q_step(0), P.dev)
    out = torch.empty(B, H, 128, device=P.dev)
    lse = torch.empty(B, H, device=P.dev)
    scratch = torch.zeros(mac.mac_workspace_size(cfg)[1], dtype=torch.uint8, device=P.dev)
    mac.mac_full_attention(cfg, scratch, q, torch.from_numpy(lens).to(P.dev), P.kv(), out, lse)
    torch.cuda.synchronize()
    st = mac.mac_last_status(cfg, scratch)
    return out, lse, st


# ---------------------------------------------------------------------------
# full attention (the miss fallback as its own call)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,Hq,Hkv,ctx,paged", [
    (BF16, 8, 2, (1, 300), False),
    (BF16, 8, 2, (129, 5000), True),
    (BF16, 4, 4, (37, 2049, 700), False),
    (BF16, 8, 4, (4096,), False),
    (F32, 4, 1, (257, 31), False),
    (F32, 2, 2, (100, 3000), True),
])
def test_full_attention_matches_oracle(dtype, Hq, Hkv, ctx, paged):
    w = W(B=len(ctx), Hq=Hq, Hkv=Hkv, ctx=ctx, dtype=dtype, steps=1)
    P = Problem(w, paged=paged)
    lens = np.array(ctx, np.int32)
    out, lse, st = full_attention_gpu(P, P.cfg(), lens)
    assert st == 0
    ref, ref_lse = O.full_attention(P.ocfg(), P.q_step(0), lens, P.okv())
    err = rel_err(out.double().cpu().numpy(), ref)
    assert err.max() <= TOL, err.max()
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=0, atol=1e-3)


def test_full_attention_long_context_ragged():
    ctx = (131072 - 5, 20000, 1)
    w = W(B=3, Hq=8, Hkv=2, ctx=ctx, steps=1, seed=3)
    P = Problem(w, device_generated=True)
    lens = np.array(ctx, np.int32)
    out, lse, st = full_attention_gpu(P, P.cfg(), lens)
    assert st == 0
    ref, ref_lse = O.full_attention(P.ocfg(), P.q_step(0), lens, P.okv())
    assert rel_err(out.double().cpu().numpy(), ref).max() <= TOL
    np.testing.assert_allclose(lse.cpu().numpy(), ref_lse, rtol=0, atol=1e-3)


# ---------------------------------------------------------------------------
# decode trajectories against the oracle
# ---------------------------------------------------------------------------

def test_tiny_config_trajectory_seeded():
    # batch 1, 1 q/1 kv head, d=128, context 4096, K=64, r=32, tau=0.6, fp32,
    # AR(1) queries with 1-in-8 jumps, 64 steps, seed 0; rings seeded with the
    # exact summaries of the last K prompt positions
    w = WORKLOADS["tiny-4k"]
    P = Problem(w, n_seed=w.ring_k)
    gpu, st, layer = gpu_trajectory(P, w.n_steps)
    ref = oracle_trajectory(P, w.n_steps)
    c = compare(gpu, ref, O.threshold_sq(128, w.tau))
    assert st == 0
    assert c["mismatched"] == 0, c
    assert c["max_err"] <= TOL, c
    assert 0 < c["hits"] < w.n_steps  # mixed hits and misses
    layer.release()


@pytest.mark.parametrize("query,tau,K,r", [
    ("clustered", 0.6, 128, 64),
    ("ar1_jump", 0.6, 64, 32),
    ("ar1_skew", 0.45, 64, 200),
    ("ar1_098", 0.75, 32, 1),
])
def test_trajectory_from_empty_rings(query, tau, K, r):
    w = W(B=2, Hq=8, Hkv=2, ctx=(3000, 5000), K=K, r=r, tau=tau, steps=48, query=query, seed=21)
    P = Problem(w)
    gpu, st, layer = gpu_trajectory(P, w.n_steps)
    ref = oracle_trajectory(P, w.n_steps)
    c = compare(gpu, ref, O.threshold_sq(128, tau))
    assert st == 0
    assert c["mismatched"] == 0, c
    assert c["max_err"] <= TOL, c
    assert c["hits"] > 0
    layer.release()


@pytest.mark.parametrize("Hq,Hkv,dtype,paged", [(4, 4, BF16, False), (8, 4, F32, False),
                                                (8, 2, BF16, True), (4, 1, F32, True),
                                                (16, 2, BF16, False), (8, 1, F32, True),
                                                (16, 2, BF16, True)])
def test_trajectory_seeded_gqa_dtypes(Hq, Hkv, dtype, paged):
    w = W(B=2, Hq=Hq, Hkv=Hkv, ctx=(900, 2000), K=32, r=16, dtype=dtype, steps=24,
          query="ar1_skew", tau=0.45, seed=5)
    P = Problem(w, n_seed=32, paged=paged)
    gpu, st, layer = gpu_trajectory(P, w.n_steps)
    ref = oracle_trajectory(P, w.n_steps)
    c = compare(gpu, ref, O.threshold_sq(128, w.tau))
    assert st == 0 and c["mismatched"] == 0 and c["max_err"] <= TOL, c
    layer.release()


def test_edge_lengths_and_band_wider_than_context():
    # m from 1 upwards (first tokens: empty candidate windows, band r >= m,
    # K > m), several tail-chunk boundaries, and r = 0 in a second run
    w = W(B=3, Hq=4, Hkv=2, ctx=(0, 127, 255), K=300, r=130, steps=40, seed=9,
          query="ar1_098", tau=0.75)
    P = Problem(w)
    gpu, st, layer = gpu_trajectory(P, w.n_steps)
    ref = oracle_trajectory(P, w.n_steps)
    c = compare(gpu, ref, O.threshold_sq(128, w.tau))
    assert st == 0 and c["mismatched"] == 0 and c["max_err"] <= TOL, c
    layer.release()
    gpu, st, layer = gpu_trajectory(P, w.n_steps, cfg=P.cfg(band_r=0))
    ref = oracle_trajectory(P, w.n_steps, band_r=0)
    c = compare(gpu, ref, O.threshold_sq(128, w.tau))
    assert st == 0 and c["mismatched"] == 0 and c["max_err"] <= TOL, c
    layer.release()


def test_min_context_and_threshold_mode():
    w = W(B=2, Hq=4, Hkv=1, ctx=(100, 400), K=64, r=8, steps=24, query="ar1_098", tau=0.75)
    P = Problem(w)
    for kw in (dict(min_context=300), dict(thr_mode=mac.MAC_THR_TAU)):
        okw = dict(min_context=kw.get("min_context", 0), thr_mode=kw.get("thr_mode", 0))
        gpu, st, layer = gpu_trajectory(P, w.n_steps, cfg=P.cfg(**kw))
        ref = oracle_trajectory(P, w.n_steps, **okw)
        c = compare(gpu, ref, O.threshold_sq(128, w.tau, okw["thr_mode"]))
        assert st == 0 and c["mismatched"] == 0 and c["max_err"] <= TOL, c
        layer.release()


def test_repeated_queries_reuse_is_exact_on_gpu():
    # RoPE off, queries repeating with period 5: every step after the first
    # cycle hits at m-5 and the reused output equals exact attention
    w = W(B=2, Hq=8, Hkv=2, ctx=(2000, 3333), K=64, r=3, tau=0.99, steps=30)
    P = Problem(w)
    pat = P.q[:, :, :5].copy()
    for s in range(P.q.shape[2]):
        P.q[:, :, s] = pat[:, :, (s - P.n_seed) % 5]
    cfg = P.cfg(rope_mode=mac.MAC_ROPE_NONE)
    gpu, st, layer = gpu_trajectory(P, w.n_steps, cfg=cfg)
    assert st == 0
    for s, (out, mp) in enumerate(gpu):
        m = P.m(s)
        if s >= 5:
            assert (mp == (m - 5)[:, None]).all()
        full, _ = O.full_attention(P.ocfg(rope_mode=O.ROPE_NONE), P.q_step(s), m, P.okv())
        assert rel_err(out, full).max() <= TOL
    layer.release()


@pytest.mark.parametrize("K", [64, 200])
def test_match_at_the_oldest_candidate_fused_and_aux(K):
    # Queries repeat with period exactly K (RoPE off, tau = 0.99: only an
    # identical query matches), so every hit lands on p = m - K, whose ring
    # slot is the one the step appends to (m mod K).  The fused append (no
    # auxiliary stream) must read the cached summary before overwriting it;
    # both paths must equal exact attention, the oracle, and each other.
    w = W(B=2, Hq=8, Hkv=2, ctx=(2000, 3333), K=K, r=3, tau=0.99, steps=40)
    P = Problem(w, n_seed=K)
    pat = P.q[:, :, :K].copy()
    for i in range(P.q.shape[2]):
        P.q[:, :, i] = pat[:, :, i % K]
    cfg = P.cfg(rope_mode=mac.MAC_ROPE_NONE)
    fused, st_f, lf = gpu_trajectory(P, w.n_steps, cfg=cfg)
    aux, st_a, la = gpu_trajectory(P, w.n_steps, cfg=cfg, aux=True)
    assert st_f == 0 and st_a == 0
    ocfg = P.ocfg(rope_mode=O.ROPE_NONE)
    for s, ((of, pf), (oa, pa)) in enumerate(zip(fused, aux)):
        m = P.m(s)
        assert (pf == (m - K)[:, None]).all()
        assert np.array_equal(pf, pa) and np.array_equal(of, oa)
        full, _ = O.full_attention(ocfg, P.q_step(s), m, P.okv())
        assert rel_err(of, full).max() <= TOL
    ref = oracle_trajectory(P, w.n_steps, rope_mode=O.ROPE_NONE)
    c = compare(fused, ref, O.threshold_sq(128, w.tau))
    assert c["mismatched"] == 0 and c["max_err"] <= TOL, c
    lf.release()
    la.release()


@pytest.mark.parametrize("F,seeded,paged,Hq,Hkv,dtype", [
    (64, True, False, 8, 2, BF16), (128, False, False, 8, 2, BF16), (100, True, True, 4, 1, BF16),
    (3000, True, False, 8, 8, BF16), (96, True, False, 8, 4, F32), (40, False, True, 4, 4, F32),
])
def test_front_sink_trajectory(F, seeded, paged, Hq, Hkv, dtype):
    # front-sink isolation ([MAC] "Production version"): the reused summaries
    # leave out [1, F] and every step attends it exactly; F = 3000 also
    # exceeds the shorter request's context (all sink, no summary)
    w = W(B=2, Hq=Hq, Hkv=Hkv, ctx=(2500, 6000), K=64, r=32, steps=32, query="ar1_skew", tau=0.45,
          seed=31, dtype=dtype)
    P = Problem(w, n_seed=64 if seeded else 0, paged=paged)
    gpu, st, layer = gpu_trajectory(P, w.n_steps, cfg=P.cfg(front_sink=F))
    ref = oracle_trajectory(P, w.n_steps, front_sink=F)
    c = compare(gpu, ref, O.threshold_sq(128, w.tau))
    assert st == 0 and c["mismatched"] == 0 and c["max_err"] <= TOL, c
    assert c["hits"] > 0
    layer.release()


def test_front_sink_repeated_queries_stay_exact():
    # RoPE off and queries repeating with period 5: each hit reuses a summary
    # of [F+1, p-r] and attends the sink afresh, so the output is exact
    # attention (a sink counted twice, or dropped, would show here)
    w = W(B=2, Hq=8, Hkv=2, ctx=(2000, 3333), K=64, r=3, tau=0.99, steps=30)
    P = Problem(w)
    pat = P.q[:, :, :5].copy()
    for s in range(P.q.shape[2]):
        P.q[:, :, s] = pat[:, :, (s - P.n_seed) % 5]
    cfg = P.cfg(rope_mode=mac.MAC_ROPE_NONE, front_sink=128)
    gpu, st, layer = gpu_trajectory(P, w.n_steps, cfg=cfg)
    assert st == 0
    for s, (out, mp) in enumerate(gpu):
        m = P.m(s)
        if s >= 5:
            assert (mp == (m - 5)[:, None]).all()
        full, _ = O.full_attention(P.ocfg(rope_mode=O.ROPE_NONE), P.q_step(s), m, P.okv())
        assert rel_err(out, full).max() <= TOL
    layer.release()


# ---------------------------------------------------------------------------
# bitwise self-consistency
# ---------------------------------------------------------------------------

def test_miss_path_bitwise_equals_full_attention():
    # empty rings: every head misses, so the decode output must be the
    # full-attention output bit for bit (same chunks, same merge order)
    w = W(B=3, Hq=8, Hkv=2, ctx=(50, 4097, 20000), steps=1)
    P = Problem(w)
    cfg = P.cfg()
    gpu, st, layer = gpu_trajectory(P, 1, cfg=cfg)
    full, _, st2 = full_attention_gpu(P, cfg, P.m(0))
    assert st == 0 and st2 == 0
    assert (gpu[0][1] == -1).all()
    assert np.array_equal(gpu[0][0], full.double().cpu().numpy())
    layer.release()


def test_paged_equals_contiguous():
    # The same cache, contiguous and paged: identical decisions, and outputs
    # that differ only in summation order (a contiguous tile starts at its
    # piece's first token, a paged one at that token's page), far inside
    # the parity tolerance.
    w = W(B=2, Hq=8, Hkv=2, ctx=(1000, 2500), K=64, r=32, steps=20, query="ar1_skew", tau=0.45)
    a, st_a, la = gpu_trajectory(Problem(w, n_seed=64), w.n_steps)
    b, st_b, lb = gpu_trajectory(Problem(w, n_seed=64, paged=True), w.n_steps)
    assert st_a == 0 and st_b == 0
    for (oa, pa), (ob, pb) in zip(a, b):
        assert np.array_equal(pa, pb)
        assert rel_err(oa, ob).max() <= 1e-5
    la.release()
    lb.release()


def test_deterministic_aux_stream_and_graph_capture():
    w = W(B=2, Hq=8, Hkv=2, ctx=(1500, 2600), K=64, r=32, steps=16, query="clustered")
    P = Problem(w, n_seed=40)
    base, st0, l0 = gpu_trajectory(P, w.n_steps)
    again, st1, l1 = gpu_trajectory(P, w.n_steps)
    aux, st2, l2 = gpu_trajectory(P, w.n_steps, aux=True)
    graph, st3, l3 = gpu_trajectory(P, w.n_steps, aux=True, graph=True)
    assert st0 == st1 == st2 == st3 == 0
    for run in (again, aux, graph):
        for (oa, pa), (ob, pb) in zip(base, run):
            assert np.array_equal(pa, pb)
            assert np.array_equal(oa, ob)
    for layer in (l0, l1, l2, l3):
        layer.release()


# ---------------------------------------------------------------------------
# device status word: bad inputs are skipped and reported, never faulted on
# ---------------------------------------------------------------------------

def test_status_reports_bad_page_and_bad_length():
    w = W(B=2, Hq=4, Hkv=2, ctx=(200, 300), steps=1)
    P = Problem(w, paged=True)
    cfg = P.cfg()
    table = P.table_dev.clone()
    table[1, 3] = 10 ** 6  # page id beyond the pool (checked before any copy)
    kv = mac.kv_view(P.kp_dev, P.vp_dev, table)
    q = to_dev(P.q_step(0), P.dev)
    out = torch.empty(2, 4, 128, device=P.dev)
    scratch = torch.zeros(mac.mac_workspace_size(cfg)[1], dtype=torch.uint8, device=P.dev)
    mac.mac_full_attention(cfg, scratch, q, torch.from_numpy(P.m(0)).to(P.dev), kv, out)
    assert mac.mac_last_status(cfg, scratch) & mac.MAC_DEV_BAD_PAGE
    assert mac.mac_last_status(cfg, scratch) == 0  # reading clears it
    too_long = np.array([P.cap + 1, 5], np.int32)
    layer = mac.MacLayer(cfg, device=P.dev)
    mac.mac_init_rings(cfg, layer.ring, layer.scratch, None, None, 0, None)
    mp = torch.empty(2, 4, dtype=torch.int32, device=P.dev)
    mac.mac_decode_step(cfg, layer.ring, layer.scratch, q, torch.from_numpy(too_long).to(P.dev),
                        P.kv(), out, mp)
    assert mac.mac_last_status(cfg, layer.scratch) & mac.MAC_DEV_BAD_SEQ_LEN
    o = out.cpu().numpy()
    assert (o[0] == 0).all() and np.isfinite(o[1]).all()
    layer.release()
