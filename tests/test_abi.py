"""The C ABI without a GPU: the library loads, exports every function
include/mac.h declares, sizes workspaces, validates arguments, and computes
the same threshold as the oracle (two independent implementations)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT, read_golden


@pytest.fixture(scope="module")
def mac():
    from long_context_decode_gb300 import build as b
    b.build()
    from long_context_decode_gb300 import mac as m
    m.load()
    return m


def header_functions():
    src = open(os.path.join(ROOT, "include", "mac.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*[\w\s\*]+?\b(mac_\w+)\s*\(", src, flags=re.M)))


def test_every_declared_function_is_exported(mac):
    declared = header_functions()
    assert len(declared) >= 10
    lib = ctypes.CDLL(mac.lib_path())
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(mac.EXPORTS) == declared


def test_struct_sizes_match_the_header(mac):
    # mac_config: 6 int32, double, int32(+pad), double, 4 int32, int64, int32(+pad) = 80 bytes
    assert ctypes.sizeof(mac.mac_config) == 80
    assert ctypes.sizeof(mac.mac_kv) == 40
    assert ctypes.sizeof(mac.mac_ring_layout) == 72


def test_workspace_sizes_and_validation(mac):
    cfg = mac.config(4, 32, 8, max_context=131072)
    ring, scratch = mac.mac_workspace_size(cfg)
    assert ring > 0 and scratch > 0
    lay = mac.mac_ring_layout_of(cfg)
    parts = [lay.pos, lay.q, lay.o, lay.lse, lay.stage_q, lay.stage_o, lay.stage_lse, lay.ctl, lay.total]
    assert parts == sorted(parts) and all(p % 256 == 0 for p in parts)
    assert lay.total == ring
    bad = [
        (dict(batch=0, n_q_heads=32, n_kv_heads=8), mac.MAC_ERR_INVALID_ARG),
        (dict(batch=1, n_q_heads=30, n_kv_heads=8), mac.MAC_ERR_INVALID_ARG),
        (dict(batch=1, n_q_heads=32, n_kv_heads=2), mac.MAC_ERR_UNSUPPORTED),  # GQA 16
        (dict(batch=1, n_q_heads=32, n_kv_heads=8, head_dim=64), mac.MAC_ERR_UNSUPPORTED),
        (dict(batch=1, n_q_heads=32, n_kv_heads=8, page_size=8), mac.MAC_ERR_UNSUPPORTED),
        (dict(batch=1, n_q_heads=32, n_kv_heads=8, band_r=-1), mac.MAC_ERR_INVALID_ARG),
        (dict(batch=1, n_q_heads=32, n_kv_heads=8, ring_k=0), mac.MAC_ERR_INVALID_ARG),
        (dict(batch=1, n_q_heads=32, n_kv_heads=8, dtype=7), mac.MAC_ERR_INVALID_ARG),
        (dict(batch=1, n_q_heads=32, n_kv_heads=8, rope_mode=9), mac.MAC_ERR_INVALID_ARG),
        (dict(batch=1, n_q_heads=32, n_kv_heads=8, rope_base=0.0), mac.MAC_ERR_INVALID_ARG),
        (dict(batch=1024, n_q_heads=32, n_kv_heads=8), mac.MAC_ERR_UNSUPPORTED),  # > 4096 units
        (dict(batch=1, n_q_heads=32, n_kv_heads=8, front_sink=-1), mac.MAC_ERR_INVALID_ARG),
        (dict(batch=1, n_q_heads=32, n_kv_heads=8, front_sink=1 << 30), mac.MAC_ERR_UNSUPPORTED),
    ]
    lib = mac.load()
    for kw, code in bad:
        c = mac.config(**kw)
        assert lib.mac_workspace_size(ctypes.byref(c), None, None) == code, kw


def test_null_and_misaligned_arguments_are_rejected_before_any_launch(mac):
    lib = mac.load()
    cfg = mac.config(1, 8, 2, max_context=4096)
    kv = mac.mac_kv(16, 16, None, 4096, 0, 0)
    assert lib.mac_decode_step(ctypes.byref(cfg), None, 256, 256, 256, ctypes.byref(kv), 256, None,
                               None, None) == mac.MAC_ERR_INVALID_ARG
    assert lib.mac_decode_step(ctypes.byref(cfg), 256, 256, 258, 256, ctypes.byref(kv), 256, None,
                               None, None) == mac.MAC_ERR_INVALID_ARG  # misaligned query
    kv_bad = mac.mac_kv(16, 24, None, 4096, 0, 0)
    assert lib.mac_full_attention(ctypes.byref(cfg), 256, 256, 256, ctypes.byref(kv_bad), 256, None,
                                  None) == mac.MAC_ERR_INVALID_ARG
    paged = mac.config(1, 8, 2, page_size=16, max_context=4096)
    kv_nopt = mac.mac_kv(16, 16, None, 0, 8, 8)
    assert lib.mac_full_attention(ctypes.byref(paged), 256, 256, 256, ctypes.byref(kv_nopt), 256,
                                  None, None) == mac.MAC_ERR_INVALID_ARG
    assert lib.mac_init_rings(ctypes.byref(cfg), 256, 256, 256, None, 4, None, None) == \
        mac.MAC_ERR_INVALID_ARG
    big = mac.config(1, 8, 2, ring_k=16, max_context=4096)
    assert lib.mac_init_rings(ctypes.byref(big), 256, 256, 256, 256, 17, ctypes.byref(kv), None) == \
        mac.MAC_ERR_INVALID_ARG  # more seeds than ring slots
    assert mac.mac_status_string(mac.MAC_ERR_CUDA) == "CUDA error"
    assert mac.mac_status_string(12345) == "unknown status"


def test_threshold_matches_oracle(mac):
    from oracle import mac_oracle as O
    for tau in (0.45, 0.6, 0.75, 0.0, 0.999):
        for mode in (mac.MAC_THR_ONE_MINUS_TAU, mac.MAC_THR_TAU):
            cfg = mac.config(1, 1, 1, tau=tau, thr_mode=mode)
            assert mac.mac_threshold_sq(cfg) == O.threshold_sq(128, tau, mode)


def test_aux_memory_fraction_matches_the_pages(mac):
    # The two rings (bf16 pre-RoPE queries; fp32 normalised summaries plus an
    # fp32 ln-LSE) relative to a bf16 KV cache of the same layer.
    for ctx, K, hq, hkv, d, pct in read_golden("aux_memory_fraction.txt")["frac"]:
        cfg = mac.config(1, int(hq), int(hkv), int(d), ring_k=int(K), max_context=int(ctx))
        lay = mac.mac_ring_layout_of(cfg)
        ring_bytes = lay.stage_q - lay.q  # query ring + summary ring + LSE ring
        kv_bytes = ctx * hkv * 2 * d * 2
        assert round(100 * ring_bytes / kv_bytes, 1) == pct
