"""GPU tests of the ready gate (mac_reset_requests) and of the bounded
waits running out (mac_test_wait_budget), for the span kernel (GQA 4) and
the ring kernel (GQA 8)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from harness import TOL, Problem, compare, rel_err, to_dev  # noqa: E402
from long_context_decode_gb300 import mac  # noqa: E402
from long_context_decode_gb300.workloads import BF16, Workload  # noqa: E402
from oracle import mac_oracle as O  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_decode_gb300 import build as b
    b.build()
    mac.load()


def W(B=2, Hq=8, Hkv=2, ctx=(2000, 3333), K=64, r=16, tau=0.6, steps=10, seed=21, query="clustered"):
    return Workload("gate", B, Hq, Hkv, 128, list(ctx), K, r, tau, BF16, 0, steps, seed, query, "normal")


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (16, 2)])
def test_reset_request_misses_then_refills_inside_a_graph(Hq, Hkv):
    # One decode step captured as a graph behind mac_reset_requests; between
    # replays only device buffers change (the step's queries and lengths, and
    # the reset flags).  Request 0 is reset before step 4: that step misses on
    # all its heads and equals exact attention, request 1 is untouched, and
    # the steps after match the oracle under the same reset.
    w = W(Hq=Hq, Hkv=Hkv)
    P = Problem(w, n_seed=w.ring_k)
    cfg = P.cfg()
    layer = mac.MacLayer(cfg, device=P.dev)
    kv = P.kv()
    mac.mac_init_rings(cfg, layer.ring, layer.scratch, to_dev(P.q_seed(), P.dev), torch.from_numpy(P.L).to(P.dev),
                       P.n_seed, kv)
    B, H, d = w.batch, w.n_q_heads, w.head_dim
    q_cur = torch.empty(B, H, d, dtype=torch.bfloat16, device=P.dev)
    m_cur = torch.empty(B, dtype=torch.int32, device=P.dev)
    flags = torch.zeros(B, dtype=torch.int32, device=P.dev)
    out = torch.empty(B, H, d, device=P.dev)
    mp = torch.empty(B, H, dtype=torch.int32, device=P.dev)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(P.dev)
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            mac.mac_reset_requests(cfg, layer.ring, flags, s)
            mac.mac_decode_step(cfg, layer.ring, layer.scratch, q_cur, m_cur, kv, out, mp, s, None)
    reset_at = 4
    gpu = []
    for st in range(w.n_steps):
        q_cur.copy_(to_dev(P.q_step(st), P.dev))
        m_cur.copy_(torch.from_numpy(P.m(st)).to(P.dev))
        if st == reset_at:
            flags.copy_(torch.tensor([1, 0], dtype=torch.int32, device=P.dev))
        g.replay()
        torch.cuda.synchronize()
        gpu.append((out.double().cpu().numpy(), mp.cpu().numpy()))
    assert mac.mac_last_status(cfg, layer.scratch) == 0
    assert flags.cpu().numpy().tolist() == [0, 0]  # consumed on the device
    ocfg, okv = P.ocfg(), P.okv()
    ring = O.Ring(ocfg)
    O.seed_rings(ocfg, ring, P.q_seed(), P.L, okv)
    ref = []
    for st in range(w.n_steps):
        if st == reset_at:
            O.reset_requests(ocfg, ring, np.array([1, 0], np.int32))
        ref.append(O.decode_step(ocfg, ring, P.q_step(st), P.m(st), okv))
    c = compare(gpu, ref, O.threshold_sq(128, w.tau))
    assert c["mismatched"] == 0 and c["max_err"] <= TOL, c
    assert (gpu[reset_at][1][0] == -1).all()  # every head of the reset request misses
    full, _ = O.full_attention(ocfg, P.q_step(reset_at), P.m(reset_at), okv)
    assert rel_err(gpu[reset_at][0][0], full[0]).max() <= TOL
    assert (gpu[reset_at - 1][1] >= 1).any() and (gpu[reset_at][1][1] >= 1).any()  # hits before and beside
    layer.release()


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (16, 2)])
@pytest.mark.parametrize("mode", ["decode", "full"])
def test_a_withheld_stage_runs_the_wait_out(Hq, Hkv, mode):
    # No copy is ever issued for stage use 1: the wait for it gives up after
    # 2^16 cycles, the launch reports MAC_DEV_WAIT_TIMEOUT and returns (the
    # synchronize below finishes), and a launch on fresh scratch afterwards
    # is clean and correct.  Nothing faults: the waits are bounded and every
    # copy that was issued lands before the kernel exits.
    w = W(Hq=Hq, Hkv=Hkv, steps=1)
    P = Problem(w, n_seed=w.ring_k)
    cfg = P.cfg()
    kv = P.kv()
    B, H, d = w.batch, w.n_q_heads, w.head_dim
    q = to_dev(P.q_step(0), P.dev)
    m = torch.from_numpy(P.m(0)).to(P.dev)

    def launch(test_budget):
        layer = mac.MacLayer(cfg, device=P.dev)
        mac.mac_init_rings(cfg, layer.ring, layer.scratch, to_dev(P.q_seed(), P.dev),
                           torch.from_numpy(P.L).to(P.dev), P.n_seed, kv)
        torch.cuda.synchronize()
        out = torch.empty(B, H, d, device=P.dev)
        mp = torch.empty(B, H, dtype=torch.int32, device=P.dev)
        if test_budget:
            mac.mac_test_wait_budget(1 << 16, 1)
        if mode == "decode":
            mac.mac_decode_step(cfg, layer.ring, layer.scratch, q, m, kv, out, mp, None, None)
        else:
            mac.mac_full_attention(cfg, layer.scratch, q, m, kv, out, None)
        torch.cuda.synchronize()
        status = mac.mac_last_status(cfg, layer.scratch)
        res = out.double().cpu().numpy()
        layer.release()
        return status, res

    status, _ = launch(True)
    assert status & mac.MAC_DEV_WAIT_TIMEOUT, status
    status, res = launch(False)
    assert status == 0
    ocfg, okv = P.ocfg(), P.okv()
    if mode == "full":
        ref, _ = O.full_attention(ocfg, P.q_step(0), P.m(0), okv)
    else:
        ring = O.Ring(ocfg)
        O.seed_rings(ocfg, ring, P.q_seed(), P.L, okv)
        ref = O.decode_step(ocfg, ring, P.q_step(0), P.m(0), okv)["out"]
    assert rel_err(res, ref).max() <= TOL


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (16, 2)])
@pytest.mark.parametrize("first", ["decode", "full"])
def test_full_attention_after_a_failed_launch_on_the_same_scratch(Hq, Hkv, first):
    # A launch that fails (a withheld stage runs its wait out) may leave
    # merge counts behind in the scratch.  Full attention on the same
    # scratch, with no reset in between and the status left unread, must
    # still be exact: its counts start from zero.
    w = W(Hq=Hq, Hkv=Hkv, steps=1)
    P = Problem(w, n_seed=w.ring_k)
    cfg = P.cfg()
    kv = P.kv()
    B, H, d = w.batch, w.n_q_heads, w.head_dim
    q = to_dev(P.q_step(0), P.dev)
    m = torch.from_numpy(P.m(0)).to(P.dev)
    layer = mac.MacLayer(cfg, device=P.dev)
    mac.mac_init_rings(cfg, layer.ring, layer.scratch, to_dev(P.q_seed(), P.dev),
                       torch.from_numpy(P.L).to(P.dev), P.n_seed, kv)
    torch.cuda.synchronize()
    out = torch.empty(B, H, d, device=P.dev)
    mp = torch.empty(B, H, dtype=torch.int32, device=P.dev)
    mac.mac_test_wait_budget(1 << 16, 1)
    if first == "decode":
        mac.mac_decode_step(cfg, layer.ring, layer.scratch, q, m, kv, out, mp, None, None)
    else:
        mac.mac_full_attention(cfg, layer.scratch, q, m, kv, out, None)
    torch.cuda.synchronize()
    out2 = torch.empty(B, H, d, device=P.dev)
    mac.mac_full_attention(cfg, layer.scratch, q, m, kv, out2, None)
    torch.cuda.synchronize()
    status = mac.mac_last_status(cfg, layer.scratch)
    assert status & mac.MAC_DEV_WAIT_TIMEOUT, status  # the failed launch's report, still unread
    ref, _ = O.full_attention(P.ocfg(), P.q_step(0), P.m(0), P.okv())
    assert rel_err(out2.double().cpu().numpy(), ref).max() <= TOL
    layer.release()
