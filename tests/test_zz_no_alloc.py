"""mac_full_attention_noalloc: full attention whose scratch is a fixed array
inside the library, for callers that cannot allocate device memory (their
device memory belongs to another allocator, or an allocation could stall the
device at a bad time).  It must give what mac_full_attention gives with a
caller-allocated scratch, call after call, since consecutive calls share the
array and each one has to clear what the last one left behind."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from harness import TOL, Problem, rel_err, to_dev  # noqa: E402
from long_context_decode_gb300 import mac  # noqa: E402
from long_context_decode_gb300.workloads import BF16, F32, Workload  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from long_context_decode_gb300 import build as b
    b.build()
    mac.load()


def _problem(ctx, dtype, Hq, Hkv, seed, paged=False):
    w = Workload("noalloc", len(ctx), Hq, Hkv, 128, list(ctx), 64, 32, 0.6, dtype, 0, 1, seed,
                 "ar1_jump", "normal")
    return Problem(w, paged=paged)


def _with_scratch(P, cfg, lens):
    out = torch.empty(P.w.batch, P.w.n_q_heads, 128, device=P.dev)
    lse = torch.empty(P.w.batch, P.w.n_q_heads, device=P.dev)
    scratch = torch.zeros(mac.mac_workspace_size(cfg)[1], dtype=torch.uint8, device=P.dev)
    mac.mac_full_attention(cfg, scratch, to_dev(P.q_step(0), P.dev), torch.from_numpy(lens).to(P.dev),
                           P.kv(), out, lse)
    return out, lse


def _noalloc(P, cfg, lens):
    out = torch.full((P.w.batch, P.w.n_q_heads, 128), float("nan"), device=P.dev)
    lse = torch.full((P.w.batch, P.w.n_q_heads), float("nan"), device=P.dev)
    mac.mac_full_attention_noalloc(cfg, to_dev(P.q_step(0), P.dev), torch.from_numpy(lens).to(P.dev),
                                   P.kv(), out, lse)
    return out, lse


def test_noalloc_matches_allocating_entry_point_on_consecutive_calls():
    cases = [
        _problem((4097, 300, 77), BF16, 8, 2, seed=1),
        _problem((20000, 1), BF16, 8, 4, seed=2, paged=True),
        _problem((129, 2500), F32, 4, 1, seed=3),
    ]
    for P in cases:  # two calls in a row per case, different problems back to back
        lens = np.array(P.w.contexts, np.int32)
        cfg = P.cfg()
        a_out, a_lse = _noalloc(P, cfg, lens)
        b_out, b_lse = _with_scratch(P, cfg, lens)
        torch.cuda.synchronize()
        assert rel_err(a_out.double().cpu().numpy(), b_out.double().cpu().numpy()).max() <= TOL
        np.testing.assert_allclose(a_lse.cpu().numpy(), b_lse.cpu().numpy(), rtol=0, atol=1e-3)
    # the same problem twice in a row: the second call reuses the array
    P = cases[0]
    lens = np.array(P.w.contexts, np.int32)
    first, _ = _noalloc(P, P.cfg(), lens)
    second, _ = _noalloc(P, P.cfg(), lens)
    ref, _ = _with_scratch(P, P.cfg(), lens)
    torch.cuda.synchronize()
    for got in (first, second):
        assert rel_err(got.double().cpu().numpy(), ref.double().cpu().numpy()).max() <= TOL


def test_noalloc_rejects_configurations_beyond_the_static_array():
    big = mac.config(128, 32, 4)  # 512 (request, kv-head) units at GQA 8: ~96 MiB of window-tile partials
    assert mac.mac_workspace_size(big)[1] > mac.MAC_NOALLOC_SCRATCH_BYTES
    kv = mac.mac_kv(256, 256, None, 1 << 20, 0, 0)
    rc = mac.load().mac_full_attention_noalloc(ctypes.byref(big), 256, 256, ctypes.byref(kv), 256,
                                               None, None)
    assert rc == mac.MAC_ERR_UNSUPPORTED
