"""Plant plausible mistakes in a copy of the oracle and check the pins catch
each one.

Every mutant is a one-spot edit of ``oracle/mac_oracle.c`` (a dropped term, a
wrong sign, an off-by-one index, a transposed head map ...) compiled on the
CPU into a temporary library; tests/test_oracle_pins.py is then run against
it and must fail.  The oracle itself is never modified.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "mac_oracle.c")

# (name, [(original text, mutated text), ...]); each original must occur once.
MUTANTS = [
    ("band start one token early", [("lo = p - r + 1;", "lo = p - r;")]),
    ("tail starts one token late", [("int64_t tail_lo = m - r + 1;", "int64_t tail_lo = m - r + 2;")]),
    ("band stops before m-r", [("oc_summary(c, x->kv, b, g, q, lo, m - r, &bM",
                                "oc_summary(c, x->kv, b, g, q, lo, m - r - 1, &bM")]),
    ("logit scale 1/d", [("double scale = 1.0 / sqrt((double)d);", "double scale = 1.0 / (double)d;")]),
    ("merge drops rescale of Z", [("*accZ = *accZ * fa + xZ * fx;", "*accZ = *accZ * fa + xZ;")]),
    ("merge drops rescale of S", [("accS[i] = accS[i] * fa + xS[i] * fx;", "accS[i] = accS[i] + xS[i] * fx;")]),
    ("rope turns the other way", [("out[ia] = a * cs - b * sn;", "out[ia] = a * cs + b * sn;"),
                                  ("out[ib] = b * cs + a * sn;", "out[ib] = b * cs - a * sn;")]),
    ("rope frequency base^(-j/d)", [("pow(base, -2.0 * (double)j / (double)d)", "pow(base, -(double)j / (double)d)")]),
    ("rope angle from pos not pos-1", [("double ang = (double)(pos - 1) * w;", "double ang = (double)pos * w;")]),
    ("rope pairs swapped", [("int ia = (mode == OC_ROPE_HALF) ? j : 2 * j;",
                             "int ia = (mode == OC_ROPE_HALF) ? 2 * j : j;"),
                            ("int ib = (mode == OC_ROPE_HALF) ? j + half : 2 * j + 1;",
                             "int ib = (mode == OC_ROPE_HALF) ? 2 * j + 1 : j + half;")]),
    ("gqa head map h % Hkv", [("h = (int)(idx % Hq), g = h / G;", "h = (int)(idx % Hq), g = h % c->n_kv_heads;")]),
    ("full attention gqa map h % Hkv", [("oc_summary(c, x->kv, b, h / G, q, 1, m, &M, &Z, S);",
                                         "oc_summary(c, x->kv, b, h % c->n_kv_heads, q, 1, m, &M, &Z, S);")]),
    ("ties go to the oldest", [("(D == bestD && p > best)", "(D == bestD && p < best)")]),
    ("window admits a stale slot", [("p < m - K)", "p < m - K - 1)")]),
    ("window admits the current position", [("p > m - 1 ||", "p > m ||")]),
    ("threshold tau*sqrt(2d) by default", [("? tau : (1.0 - tau)", "? (1.0 - tau) : tau")]),
    ("threshold not strict", [("(dmin < x->thr2)", "(dmin <= x->thr2)")]),
    ("append to the next slot", [("int64_t slot = idx * K + m % K;", "int64_t slot = idx * K + (m + 1) % K;")]),
    ("seed summary one token too long", [("front_sink + 1, p - c->band_r, &x->ring->sM[slot]",
                                          "front_sink + 1, p - c->band_r + 1, &x->ring->sM[slot]")]),
    ("seed summary keeps the sink", [("(int64_t)c->front_sink + 1, p - c->band_r", "1, p - c->band_r")]),
    ("sink left out of the output", [("oc_summary(c, x->kv, b, g, q, 1, F < m ? F : m, &tM, &tZ, tS);",
                                      "oc_summary(c, x->kv, b, g, q, 1, 0, &tM, &tZ, tS);")]),
    ("summaries keep the sink on a miss", [("int64_t lo = F + 1;", "int64_t lo = 1;")]),
    ("front sink ignored everywhere", [("const int64_t F = c->front_sink;", "const int64_t F = 0;"),
                                       ("(int64_t)c->front_sink + 1, p - c->band_r", "1, p - c->band_r")]),
    ("summaries keep the sink on a hit", [("if (lo < F + 1) lo = F + 1;", "if (lo < 1) lo = 1;")]),
    ("max not tracked", [("if (l > mx) mx = l;", "")]),
    ("values read from K", [("S[i] += e * load_elem(kv->v, c->dtype, row + i);",
                             "S[i] += e * load_elem(kv->k, c->dtype, row + i);")]),
    ("bf16 decoded with the wrong shift", [("[i] << 16;", "[i] << 15;")]),
    ("paged row offset ignores the page", [("return ((page * c->n_kv_heads + g) * c->page_size",
                                            "return ((b * c->n_kv_heads + g) * c->page_size")]),
    ("hit reuses the wrong slot", [("int64_t slot = (((int64_t)b * Hq + h) * K + p % K);",
                                    "int64_t slot = (((int64_t)b * Hq + h) * K + (p + 1) % K);")]),
    ("distance drops the square", [("D += diff * diff;", "D += fabs(diff);")]),
    ("reset leaves the ring as it was", [("for (int s = 0; s < K; ++s) ring->pos[(int64_t)b * K + s] = 0;", ";")]),
]


def _run_mutant(tmpdir, idx, name, edits):
    src = open(SRC).read()
    for old, new in edits:
        assert src.count(old) == 1, f"{name}: '{old}' occurs {src.count(old)} times"
        src = src.replace(old, new)
    d = os.path.join(tmpdir, f"m{idx}")
    os.makedirs(d, exist_ok=True)
    c_path = os.path.join(d, "mac_oracle.c")
    with open(c_path, "w") as f:
        f.write(src)
    so = os.path.join(d, "libmac_oracle.so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", so,
                    c_path, "-lm", "-lpthread"], check=True, capture_output=True)
    env = dict(os.environ, MAC_ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return name, r.returncode, r.stdout[-400:]


def test_pins_catch_every_mutant(tmp_path):
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(lambda a: _run_mutant(str(tmp_path), *a),
                              [(i, n, e) for i, (n, e) in enumerate(MUTANTS)]))
    survivors = [(n, out) for n, rc, out in results if rc == 0]
    assert not survivors, "mutants not caught by the pins: " + "; ".join(n for n, _ in survivors)


def test_unmutated_copy_passes(tmp_path):
    name, rc, out = _run_mutant(str(tmp_path), 0, "identity", [])
    assert rc == 0, out
