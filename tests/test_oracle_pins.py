"""Pins of the fp64 oracle against what the pages and mathematics fix.

Every check here compares the oracle with something other than itself: a
value the pages print (tests/golden, cited there), a closed form, a library
routine the operation reduces to in a special case, brute force on tiny
inputs, or an invariant the method implies.  tests/test_oracle_mutants.py
plants plausible mistakes in the oracle source and checks that this file
catches each of them.
"""
import math

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

from conftest import read_golden
from oracle import mac_oracle as O


def f32(x):
    return np.ascontiguousarray(x, np.float32)


def tiny_cfg(**kw):
    base = dict(batch=1, n_q_heads=1, n_kv_heads=1, head_dim=8, ring_k=16, band_r=2, tau=0.5,
                rope_mode=O.ROPE_NONE, dtype=O.F32)
    base.update(kw)
    return O.Config(**base)


def kv_f32(k, v):
    k, v = f32(k), f32(v)
    return O.KV(k, v, capacity=k.shape[2])


# ---------------------------------------------------------------------------
# threshold (MAC blog, "Match (2)")
# ---------------------------------------------------------------------------

def test_threshold_worked_example():
    (d, tau, sqrt2d, thr), = read_golden("threshold_worked_example.txt")["worked"]
    assert math.sqrt(2 * d) == sqrt2d
    thr2 = O.threshold_sq(int(d), tau, O.THR_ONE_MINUS_TAU)
    assert thr2 == pytest.approx(thr * thr, rel=1e-6)
    # larger tau gives a smaller threshold (stricter matching)
    assert O.threshold_sq(128, 0.75) < O.threshold_sq(128, 0.6) < O.threshold_sq(128, 0.45)
    # the summary page's reading tau*sqrt(2d) is the other mode
    assert O.threshold_sq(128, 0.45, O.THR_TAU) == pytest.approx((0.45 * 16) ** 2, rel=1e-6)
    # the threshold is rounded once to fp32
    assert thr2 == float(np.float32(thr2))


# ---------------------------------------------------------------------------
# RoPE (MAC blog, "Match (1)")
# ---------------------------------------------------------------------------

def test_rope_worked_examples():
    for row in read_golden("rope_worked_examples.txt")["case"]:
        mode, d, base, pos = int(row[0]), int(row[1]), row[2], int(row[3])
        x = np.array(row[4:4 + d])
        want = np.array(row[4 + d:4 + 2 * d])
        got = O.rope(x, pos, base, mode)
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-13)


@pytest.mark.parametrize("mode", [O.ROPE_HALF, O.ROPE_INTERLEAVED])
def test_rope_relative_rotation_identity(mode):
    # ||x - R(D) x||^2 = 2 ||x||^2 (1 - avgcos(D)), avgcos = energy-weighted
    # mean of cos(D w_j) over the 2x2 blocks (MAC blog, "Match (1)").
    rng = np.random.default_rng(0)
    d, base = 128, 10000.0
    x = rng.standard_normal(d)
    half = d // 2
    w = base ** (-2.0 * np.arange(half) / d)
    if mode == O.ROPE_HALF:
        energy = x[:half] ** 2 + x[half:] ** 2
    else:
        energy = x[0::2] ** 2 + x[1::2] ** 2
    n2 = float(x @ x)
    for delta in [0, 1, 7, 100, 4095, 131071]:
        rx = O.rope(x, delta + 1, base, mode)  # position delta+1 rotates by delta
        lhs = float(np.sum((x - rx) ** 2))
        avgcos = float(np.sum(energy * np.cos(delta * w)) / n2)
        assert lhs == pytest.approx(2 * n2 * (1 - avgcos), rel=1e-9, abs=1e-9)


@pytest.mark.parametrize("mode", [O.ROPE_HALF, O.ROPE_INTERLEAVED])
def test_rope_group_properties(mode):
    rng = np.random.default_rng(1)
    x = rng.standard_normal(128)
    # the first position is the identity
    np.testing.assert_array_equal(O.rope(x, 1, 10000.0, mode), x)
    # rotations preserve the norm and compose additively
    for a, b in [(3, 5), (1000, 77), (65536, 65536)]:
        ra = O.rope(x, a + 1, 10000.0, mode)
        assert np.linalg.norm(ra) == pytest.approx(np.linalg.norm(x), rel=1e-13)
        np.testing.assert_allclose(O.rope(ra, b + 1, 10000.0, mode), O.rope(x, a + b + 1, 10000.0, mode),
                                   rtol=0, atol=1e-9)
    np.testing.assert_array_equal(O.rope(x, 12345, 10000.0, O.ROPE_NONE), x)


# ---------------------------------------------------------------------------
# logits, summaries and the merge (MAC blog "Decomposable attention",
# "Complete"; sharded-softmax merge on the "Attention Cache and Sequence
# Parallelism" page)
# ---------------------------------------------------------------------------

def test_logit_scale_cauchy_schwarz_tight():
    # |l_t(q1) - l_t(q2)| <= ||q1 - q2|| ||K_t|| / sqrt(d) (MAC blog "Match (1)"),
    # with equality when K_t is parallel to q1 - q2; a single-token summary has
    # M = l_t.
    rng = np.random.default_rng(2)
    d = 16
    q1, q2 = rng.standard_normal(d), rng.standard_normal(d)
    kvec = 0.7 * (q1 - q2)
    k = np.zeros((1, 1, 3, d), np.float32)
    k[0, 0, 0] = kvec
    k[0, 0, 1:] = rng.standard_normal((2, d))
    v = rng.standard_normal((1, 1, 3, d)).astype(np.float32)
    cfg, kv = tiny_cfg(head_dim=d), kv_f32(k, v)
    kk = k[0, 0].astype(np.float64)
    for t in range(3):
        l1 = O.summary(cfg, kv, 0, 0, q1, t + 1, t + 1)[0]
        l2 = O.summary(cfg, kv, 0, 0, q2, t + 1, t + 1)[0]
        bound = np.linalg.norm(q1 - q2) * np.linalg.norm(kk[t]) / math.sqrt(d)
        if t == 0:
            assert abs(l1 - l2) == pytest.approx(bound, rel=1e-12)
        else:
            assert abs(l1 - l2) <= bound * (1 + 1e-12)


def test_summary_matches_softmax_library():
    rng = np.random.default_rng(3)
    d, n = 32, 200
    k = rng.standard_normal((1, 1, n, d)).astype(np.float32) * 3
    v = rng.standard_normal((1, 1, n, d)).astype(np.float32)
    q = rng.standard_normal(d)
    cfg, kv = tiny_cfg(head_dim=d), kv_f32(k, v)
    M, Z, S = O.summary(cfg, kv, 0, 0, q, 1, n)
    logits = (k[0, 0].astype(np.float64) @ q) / math.sqrt(d)
    np.testing.assert_allclose(S / Z, softmax(logits) @ v[0, 0].astype(np.float64), rtol=1e-12)
    assert M + math.log(Z) == pytest.approx(logsumexp(logits), rel=1e-13)
    assert M == pytest.approx(logits.max(), rel=1e-15)
    # empty range is the empty summary
    M0, Z0, S0 = O.summary(cfg, kv, 0, 0, q, 5, 4)
    assert M0 == -np.inf and Z0 == 0 and not S0.any()


def test_merge_associativity_random_partitions():
    # summaries of disjoint sets combine to the summary of the union in any
    # grouping and order; splitting at p = m-1 and adding one token at a time
    # is the online-softmax recurrence
    rng = np.random.default_rng(4)
    d, n = 16, 97
    k = (rng.standard_normal((1, 1, n, d)) * 4).astype(np.float32)
    v = rng.standard_normal((1, 1, n, d)).astype(np.float32)
    q = rng.standard_normal(d)
    cfg, kv = tiny_cfg(head_dim=d), kv_f32(k, v)
    M, Z, S = O.summary(cfg, kv, 0, 0, q, 1, n)
    ref_o, ref_lse = S / Z, M + math.log(Z)
    empty = (-np.inf, 0.0, np.zeros(d))
    for trial in range(20):
        cuts = np.sort(rng.choice(np.arange(2, n + 1), size=rng.integers(1, 12), replace=False))
        bounds = [1, *cuts.tolist(), n + 1]
        parts = [O.summary(cfg, kv, 0, 0, q, bounds[i], bounds[i + 1] - 1) for i in range(len(bounds) - 1)]
        rng.shuffle(parts)
        acc = empty
        for p in parts:
            acc = O.merge(acc, p)
        np.testing.assert_allclose(acc[2] / acc[1], ref_o, rtol=1e-12, atol=1e-14)
        assert acc[0] + math.log(acc[1]) == pytest.approx(ref_lse, rel=1e-13)
    acc = empty
    for t in range(1, n + 1):
        acc = O.merge(acc, O.summary(cfg, kv, 0, 0, q, t, t))
    np.testing.assert_allclose(acc[2] / acc[1], ref_o, rtol=1e-12, atol=1e-14)
    # the empty summary is the identity on both sides
    one = O.summary(cfg, kv, 0, 0, q, 3, 9)
    for a, b in [(O.merge(empty, one), one), (O.merge(one, empty), one)]:
        assert a[0] == b[0] and a[1] == b[1]
        np.testing.assert_array_equal(a[2], b[2])


def test_merge_handles_large_logit_gaps():
    # running-max form: no overflow even when the parts' maxima differ by 1e3
    d = 4
    a = (1000.0, 2.0, np.ones(d) * 2.0)
    b = (-5.0, 1.0, np.ones(d))
    M, Z, S = O.merge(a, b)
    assert M == 1000.0 and Z == pytest.approx(2.0) and np.all(np.isfinite(S))


# ---------------------------------------------------------------------------
# full attention and the GQA head map ("Attention Cache and Sequence
# Parallelism", MHA decode pseudo-code: scores = q K^T * scale, repeat_kv)
# ---------------------------------------------------------------------------

def test_full_attention_textbook_gqa():
    rng = np.random.default_rng(5)
    B, Hq, Hkv, d = 2, 4, 2, 16
    lens = np.array([13, 29], np.int32)
    cap = 32
    k = (rng.standard_normal((B, Hkv, cap, d)) * 2).astype(np.float32)
    v = rng.standard_normal((B, Hkv, cap, d)).astype(np.float32)
    q = rng.standard_normal((B, Hq, d)).astype(np.float32)
    cfg = tiny_cfg(batch=B, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=d, rope_mode=O.ROPE_NONE)
    out, lse = O.full_attention(cfg, q, lens, kv_f32(k, v))
    for b in range(B):
        for h in range(Hq):
            g = h // (Hq // Hkv)  # repeat_kv: consecutive q heads share a KV head
            kk = k[b, g, :lens[b]].astype(np.float64)
            logits = kk @ q[b, h].astype(np.float64) / math.sqrt(d)
            np.testing.assert_allclose(out[b, h], softmax(logits) @ v[b, g, :lens[b]], rtol=1e-12)
            assert lse[b, h] == pytest.approx(logsumexp(logits), rel=1e-13)


def test_full_attention_rotates_query_at_current_position():
    rng = np.random.default_rng(6)
    d, m = 16, 21
    k = rng.standard_normal((1, 1, m, d)).astype(np.float32)
    v = rng.standard_normal((1, 1, m, d)).astype(np.float32)
    q = rng.standard_normal((1, 1, d)).astype(np.float32)
    cfg = tiny_cfg(head_dim=d, rope_mode=O.ROPE_HALF)
    out, _ = O.full_attention(cfg, q, np.array([m], np.int32), kv_f32(k, v))
    qr = O.rope(q[0, 0].astype(np.float64), m, 10000.0, O.ROPE_HALF)
    logits = k[0, 0].astype(np.float64) @ qr / math.sqrt(d)
    np.testing.assert_allclose(out[0, 0], softmax(logits) @ v[0, 0], rtol=1e-12)


def test_bf16_inputs_decode_exactly():
    # bf16 is the upper half of an IEEE binary32: 0x3F80 = 1, 0xC000 = -2,
    # 0x3E80 = 0.25, 0x4049 = 3.140625; a one-token cache returns V exactly.
    d = 4
    v_bits = np.array([0x3F80, 0xC000, 0x3E80, 0x4049], np.uint16).reshape(1, 1, 1, d)
    k_bits = np.array([0x3F80, 0x3F80, 0x3F80, 0x3F80], np.uint16).reshape(1, 1, 1, d)
    q_bits = np.array([0x3F80, 0, 0, 0], np.uint16).reshape(1, 1, d)
    cfg = tiny_cfg(head_dim=d, dtype=O.BF16)
    out, lse = O.full_attention(cfg, q_bits, np.array([1], np.int32), O.KV(k_bits, v_bits, capacity=1))
    np.testing.assert_array_equal(out[0, 0], [1.0, -2.0, 0.25, 3.140625])
    assert lse[0, 0] == pytest.approx(1.0 / 2.0)  # l = q.k / sqrt(4) = 0.5


def test_paged_cache_reads_the_same_tokens():
    rng = np.random.default_rng(7)
    B, H, d, ps, ppr = 2, 2, 8, 4, 5
    cap = ps * ppr
    k = rng.standard_normal((B, H, cap, d)).astype(np.float32)
    v = rng.standard_normal((B, H, cap, d)).astype(np.float32)
    q = rng.standard_normal((B, H, d)).astype(np.float32)
    lens = np.array([cap, 11], np.int32)
    table = rng.permutation(B * ppr).astype(np.int32).reshape(B, ppr)
    kp = np.empty((B * ppr, H, ps, d), np.float32)
    vp = np.empty_like(kp)
    for b in range(B):
        for j in range(ppr):
            kp[table[b, j]] = k[b, :, j * ps:(j + 1) * ps]
            vp[table[b, j]] = v[b, :, j * ps:(j + 1) * ps]
    c0 = tiny_cfg(batch=B, n_q_heads=H, n_kv_heads=H, head_dim=d)
    c1 = tiny_cfg(batch=B, n_q_heads=H, n_kv_heads=H, head_dim=d, page_size=ps)
    o0, l0 = O.full_attention(c0, q, lens, kv_f32(k, v))
    o1, l1 = O.full_attention(c1, q, lens, O.KV(kp, vp, table, max_pages=ppr))
    np.testing.assert_array_equal(o0, o1)
    np.testing.assert_array_equal(l0, l1)


# ---------------------------------------------------------------------------
# match (MAC blog "Match (2)", "Match (3)", K1 pseudo-code)
# ---------------------------------------------------------------------------

def _ring_with(cfg, m, entries):
    """Ring for one request/head with (pos, query) entries at slot pos mod K."""
    ring = O.Ring(cfg)
    for pos, qv in entries:
        s = pos % cfg.ring_k
        ring.pos[0, s] = pos
        ring.q[0, 0, s] = qv
    return ring


def _step(cfg, ring, qt, m, kv):
    return O.decode_step(cfg, ring, f32(qt).reshape(1, 1, -1), np.array([m], np.int32), kv, n_threads=1)


def _kv_for(cfg, m, seed=0):
    rng = np.random.default_rng(seed)
    shape = (cfg.batch, cfg.n_kv_heads, m + 4, cfg.head_dim)
    return kv_f32(rng.standard_normal(shape), rng.standard_normal(shape))


def test_match_brute_force_tiny_rings():
    rng = np.random.default_rng(8)
    d, K = 8, 16
    cfg = tiny_cfg(head_dim=d, ring_k=K, tau=-10.0)  # threshold far above every distance
    for trial in range(50):
        m = int(rng.integers(2, 60))
        n = int(rng.integers(1, K + 1))
        cands = sorted(set(int(p) for p in rng.integers(max(1, m - K), m, size=n)))
        qs = {p: rng.standard_normal(d).astype(np.float32) for p in cands}
        qt = rng.standard_normal(d).astype(np.float32)
        ring = _ring_with(cfg, m, [(p, qs[p]) for p in cands])
        res = _step(cfg, ring, qt, m, _kv_for(cfg, m))
        dist = sorted((float(np.sum((qt.astype(np.float64) - qs[p]) ** 2)), -p) for p in cands)
        assert res["match_pos"][0, 0] == -dist[0][1]
        assert res["dmin"][0, 0] == pytest.approx(dist[0][0], rel=1e-14)
        if len(dist) > 1:
            assert res["dsecond"][0, 0] == pytest.approx(dist[1][0], rel=1e-14)


def test_match_threshold_is_strict_and_two_sided():
    d = 8
    cfg = tiny_cfg(head_dim=d, ring_k=8, tau=0.5)  # thr = 0.5 * sqrt(16) = 2, thr^2 = 4 exactly
    assert O.threshold_sq(d, 0.5) == 4.0
    m = 10
    qt = np.zeros(d, np.float32)
    kv = _kv_for(cfg, m)
    for dist, hit in [(2.0, False), (1.999, True), (2.001, False), (0.0, True)]:
        cand = np.zeros(d, np.float32)
        cand[3] = dist
        ring = _ring_with(cfg, m, [(m - 3, cand)])
        res = _step(cfg, ring, qt, m, kv)
        assert (res["match_pos"][0, 0] == m - 3) == hit, dist


def test_match_ties_go_to_most_recent():
    d = 8
    cfg = tiny_cfg(head_dim=d, ring_k=8, tau=0.0)
    m = 20
    qt = np.zeros(d, np.float32)
    a = np.zeros(d, np.float32); a[0] = 1.0
    b = np.zeros(d, np.float32); b[0] = -1.0
    for older, newer in [(13, 17), (18, 14)]:
        lo, hi = min(older, newer), max(older, newer)
        ring = _ring_with(cfg, m, [(older, a), (newer, b)])
        res = _step(cfg, ring, qt, m, _kv_for(cfg, m))
        assert res["match_pos"][0, 0] == hi
        assert res["dsecond"][0, 0] == res["dmin"][0, 0]


def test_match_window_excludes_stale_future_and_empty_slots():
    d, K = 8, 8
    cfg = tiny_cfg(head_dim=d, ring_k=K, tau=0.0)
    m = 30
    qt = np.full(d, 0.5, np.float32)
    near = qt.copy()
    far = qt + 1.0
    kv = _kv_for(cfg, m)
    # a perfect match at the oldest in-window position m-K is accepted ...
    res = _step(cfg, _ring_with(cfg, m, [(m - K, near), (m - 1, far)]), qt, m, kv)
    assert res["match_pos"][0, 0] == m - K
    # ... one step older is stale; a slot holding position m or later is not a
    # candidate either; an empty slot (position 0) is never a candidate
    for bad in [m - K - 1, m, m + K - 1]:
        ring = _ring_with(cfg, m, [(bad, near), (m - 2, far)])
        res = _step(cfg, ring, qt, m, kv)
        assert res["match_pos"][0, 0] == m - 2, bad
    ring = O.Ring(cfg)
    ring.q[0, 0, :] = near
    res = _step(cfg, ring, qt, m, kv)
    assert res["match_pos"][0, 0] == -1 and res["dmin"][0, 0] == np.inf


def test_min_context_disables_reuse():
    d = 8
    cfg = tiny_cfg(head_dim=d, ring_k=8, tau=0.0, min_context=31)
    qt = np.zeros(d, np.float32)
    kv = _kv_for(cfg, 31)
    assert _step(cfg, _ring_with(cfg, 30, [(29, qt)]), qt, 30, kv)["match_pos"][0, 0] == -1
    assert _step(cfg, _ring_with(cfg, 31, [(30, qt)]), qt, 31, kv)["match_pos"][0, 0] == 30


# ---------------------------------------------------------------------------
# miss, r >= m and reuse with an unchanged query
# ---------------------------------------------------------------------------

def _rand_problem(seed, B=2, Hq=4, Hkv=2, d=16, cap=96, rope=O.ROPE_HALF, **kw):
    rng = np.random.default_rng(seed)
    k = (rng.standard_normal((B, Hkv, cap, d)) * 2).astype(np.float32)
    v = rng.standard_normal((B, Hkv, cap, d)).astype(np.float32)
    cfg = tiny_cfg(batch=B, n_q_heads=Hq, n_kv_heads=Hkv, head_dim=d, rope_mode=rope, **kw)
    return rng, cfg, kv_f32(k, v)


@pytest.mark.parametrize("F", [0, 2, 30])
def test_miss_equals_full_attention(F):
    # an empty ring misses everywhere and the step is exact attention
    # (MAC blog "Match (1)": a miss falls back to full attention); a front
    # sink only splits [1, m] into sink, band and tail
    rng, cfg, kv = _rand_problem(9, ring_k=8, band_r=5, front_sink=F)
    for lens in ([40, 77], [3, 5], [1, 2]):
        lens = np.array(lens, np.int32)
        q = rng.standard_normal((2, 4, 16)).astype(np.float32)
        res = O.decode_step(cfg, O.Ring(cfg), q, lens, kv)
        full, _ = O.full_attention(cfg, q, lens, kv)
        assert (res["match_pos"] == -1).all()
        np.testing.assert_allclose(res["out"], full, rtol=1e-12, atol=1e-15)


def test_band_covering_context_gives_full_attention():
    # r >= m: the cached part AS_{1:p-r} is empty and the fresh range is
    # [1, m], so even a hit is exact attention (the rho -> 1 limit of "Amend")
    rng, cfg, kv = _rand_problem(10, ring_k=32, band_r=64, tau=-100.0)
    ring = O.Ring(cfg)
    lens0 = np.array([20, 31], np.int32)
    for step in range(12):
        lens = lens0 + step
        q = rng.standard_normal((2, 4, 16)).astype(np.float32)
        res = O.decode_step(cfg, ring, q, lens, kv)
        full, _ = O.full_attention(cfg, q, lens, kv)
        if step > 0:
            assert (res["match_pos"] >= 1).all()
        np.testing.assert_allclose(res["out"], full, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("K,r,cycle,seeded,F", [
    (8, 2, 1, True, 0), (8, 2, 3, False, 0), (16, 1, 5, True, 0), (16, 7, 5, False, 0), (4, 9, 3, True, 0),
    (32, 3, 11, False, 0), (6, 4, 6, True, 0),
    (8, 2, 3, True, 4), (16, 7, 5, False, 10), (6, 4, 6, True, 25), (8, 2, 1, False, 60),
])
def test_reuse_with_repeated_queries_is_exact(K, r, cycle, seeded, F):
    # With RoPE off and the query at m equal to the one stored at p, the
    # logits of [1, p-r] under q_m are exactly those under q_p (delta_t = 0 in
    # MAC blog "Reuse"), so cached (+) band (+) tail must equal exact attention.
    # Queries repeat with period `cycle`; the match lands at m - cycle, so the
    # band, tail, slot addressing and chained rectified summaries are all used.
    # With a front sink F the summaries leave out [1, F] and the sink is
    # attended at each step ([MAC] "Production version"), so the output is
    # still exact attention; F = 60 also exceeds the early steps' lengths.
    rng, cfg, kv = _rand_problem(11 + K + r + cycle, ring_k=K, band_r=r, rope=O.ROPE_NONE,
                                 tau=0.99, cap=160, front_sink=F)  # only identical queries match
    B, Hq, d = cfg.batch, cfg.n_q_heads, cfg.head_dim
    pattern = rng.standard_normal((B, Hq, cycle, d)).astype(np.float32)
    L = np.array([30, 47], np.int32)
    ring = O.Ring(cfg)
    if seeded:
        n_seed = min(K, 12)
        seeds = np.stack([pattern[:, :, (L[b] - n_seed + 1 + np.arange(n_seed)) % cycle][b]
                          for b in range(B)])
        O.seed_rings(cfg, ring, f32(seeds), L, kv)
    hits = 0
    for step in range(40):
        m = L + 1 + step
        q = np.stack([pattern[b, :, m[b] % cycle] for b in range(B)])
        res = O.decode_step(cfg, ring, f32(q), m.astype(np.int32), kv)
        full, _ = O.full_attention(cfg, f32(q), m.astype(np.int32), kv)
        np.testing.assert_allclose(res["out"], full, rtol=1e-11, atol=1e-14)
        if cycle <= K and (seeded or step >= cycle):
            for b in range(B):
                assert (res["match_pos"][b] == m[b] - cycle).all()
            hits += 1
    assert hits >= 20


@pytest.mark.parametrize("rope", [O.ROPE_NONE, O.ROPE_HALF, O.ROPE_INTERLEAVED])
def test_front_sink_covering_the_reused_prefix_gives_exact_attention(rope):
    # Front-sink isolation ([MAC] "Production version"): the reused summaries
    # cover [F+1, p-r] only and the sink [1, F] is attended afresh at every
    # step.  When F >= p - r for every hit, no reused summary holds a token,
    # so each step is exact attention under its own query although the
    # queries differ from step to step and every head hits.  An oracle that
    # dropped F would reuse the summary of [1, p-r] made with q_p.
    rng, cfg, kv = _rand_problem(13, ring_k=4, band_r=3, tau=-10.0, rope=rope, front_sink=40)
    B, Hq, d = cfg.batch, cfg.n_q_heads, cfg.head_dim
    L = np.array([35, 38], np.int32)
    ring = O.Ring(cfg)
    O.seed_rings(cfg, ring, rng.standard_normal((B, Hq, 4, d)).astype(np.float32), L, kv)
    band_tokens = 0
    for step in range(6):
        m = (L + 1 + step).astype(np.int32)
        assert (m - 1 <= 40 + 3).all()  # every candidate p <= m-1 has p - r <= F
        q = rng.standard_normal((B, Hq, d)).astype(np.float32)
        res = O.decode_step(cfg, ring, q, m, kv)
        assert (res["match_pos"] >= 1).all() and (res["match_pos"] - 3 >= 1).all()
        full, _ = O.full_attention(cfg, q, m, kv)
        np.testing.assert_allclose(res["out"], full, rtol=1e-11, atol=1e-14)
        band_tokens += int(np.maximum(0, m - 3 - 40).sum())
    assert band_tokens > 0  # the band [F+1, m-r] is attended at least once


def test_a_reset_request_misses_at_its_next_step():
    # Ready gate ([MAC] "Production version"): a reset request has no
    # candidate at its next step, so every head misses and the step is exact
    # attention; the other request is untouched, and at the step after, the
    # reset step's own append is the request's only candidate.
    rng, cfg, kv = _rand_problem(14, ring_k=4, band_r=3, tau=-10.0)
    B, Hq, d = cfg.batch, cfg.n_q_heads, cfg.head_dim
    L = np.array([30, 34], np.int32)
    ring = O.Ring(cfg)
    O.seed_rings(cfg, ring, rng.standard_normal((B, Hq, 4, d)).astype(np.float32), L, kv)
    q0, q1 = (rng.standard_normal((B, Hq, d)).astype(np.float32) for _ in range(2))
    m = (L + 1).astype(np.int32)
    kept = ring.copy()
    r_kept = O.decode_step(cfg, kept, q0, m, kv)
    assert (r_kept["match_pos"] >= 1).all()  # every head would hit
    O.reset_requests(cfg, ring, np.array([1, 0], np.int32))
    res = O.decode_step(cfg, ring, q0, m, kv)
    assert (res["match_pos"][0] == -1).all()
    full, _ = O.full_attention(cfg, q0, m, kv)
    np.testing.assert_allclose(res["out"][0], full[0], rtol=1e-11, atol=1e-14)
    np.testing.assert_array_equal(res["match_pos"][1], r_kept["match_pos"][1])
    np.testing.assert_array_equal(res["out"][1], r_kept["out"][1])
    nxt = O.decode_step(cfg, ring, q1, m + 1, kv)
    assert (nxt["match_pos"][0] == m[0]).all()


def test_seed_positions_and_slots():
    rng, cfg, kv = _rand_problem(12, ring_k=8, band_r=3)
    L = np.array([5, 40], np.int32)
    seeds = rng.standard_normal((2, 4, 8, 16)).astype(np.float32)
    ring = O.Ring(cfg)
    ring.pos[:] = 999
    O.seed_rings(cfg, ring, seeds, L, kv)
    # request 0 has only 5 prompt positions: seeds 1..5 land, the rest are skipped
    assert sorted(ring.pos[0][ring.pos[0] > 0].tolist()) == [1, 2, 3, 4, 5]
    assert sorted(ring.pos[1].tolist()) == list(range(33, 41))
    for p in range(33, 41):
        s = p % 8
        np.testing.assert_array_equal(ring.q[1, 2, s], seeds[1, 2, p - 33])
    # position 2 with r=3 has an empty rectified summary AS_{1:-1}
    assert ring.sZ[0, 0, 2 % 8] == 0.0 and ring.sM[0, 0, 2 % 8] == -np.inf
