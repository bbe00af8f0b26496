"""Planted mistakes in the oracle are caught by its pins.

Each case below copies oracle/gs_oracle.c, plants one plausible mistake (a
dropped term, a wrong sign, an open or closed bin edge, a wrong index or
ordering), builds the copy and runs the pins of tests/test_oracle_pins.py and
tests/test_oracle_six.py against it. Every copy must fail at least one pin.
The unchanged source, built and run the same way, must pass them all.

Several mistakes sit in helpers that the hub loops and the brute forces share
(the pair rule, the bin search, the clique volume). Comparing the oracle with
itself cannot catch those. Only the independent pins can: the NumPy brute
force, the hand-derived fixtures and the closed forms.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "gs_oracle.c")
PINS = ["tests/test_oracle_pins.py", "tests/test_oracle_six.py"]

# (name, text in gs_oracle.c, replacement); each text occurs exactly once
MUTANTS = [
    # pair rule and bins (GRAMSCI v2 §II.1)
    ("minimum image wraps one way only",
     "        else if (2 * d < -box) d += box;\n", ""),
    ("upper bin edge closed",
     "if (lo * lo <= d2 && d2 < hi * hi) return k;", "if (lo * lo <= d2 && d2 <= hi * hi) return k;"),
    ("lower bin edge open",
     "if (lo * lo <= d2 && d2 < hi * hi) return k;", "if (lo * lo < d2 && d2 < hi * hi) return k;"),
    ("a point is its own neighbour",
     "    if (a == b) return -1;\n    int64_t d2 = dist2(c, a, b);", "    int64_t d2 = dist2(c, a, b);"),
    ("rows filled in descending order",
     "    for (int64_t j = 0; j < g->c.n; ++j) {          /* j ascending: rows come out sorted */",
     "    for (int64_t j = g->c.n - 1; j >= 0; --j) {"),
    # 3pCF (§II.2)
    ("spokes below the hub counted too",
     "        if (j <= i) continue;                      /* spoke j > hub i */\n", ""),
    ("hub bin of k taken for j",
     "int v[3] = { t->bin[a], t->bin[b], bjk };\n            sort3(v);\n            h[t->t3[((size_t)v[0] * nb + v[1]) * nb + v[2]]] += 1;",
     "int v[3] = { t->bin[a], t->bin[a], bjk };\n            sort3(v);\n            h[t->t3[((size_t)v[0] * nb + v[1]) * nb + v[2]]] += 1;"),
    ("closing side not tested in the brute force",
     "            int bjk = pair_bin(&b->c, j, k);\n            if (bjk < 0) continue;\n            int v[3] = { bij, bik, bjk };",
     "            int bjk = pair_bin(&b->c, j, k);\n            if (bjk < 0) bjk = 0;\n            int v[3] = { bij, bik, bjk };"),
    # parity 4pCF (§III.1.1, §III.2 Eq.(3))
    ("cross product term with the wrong sign",
     "int64_t cy = r1[2] * r2[0] - r1[0] * r2[2];", "int64_t cy = r1[0] * r2[2] - r1[2] * r2[0];"),
    ("volume taken in row order, not bin order",
     "displacement(c, hub, s[order[q]], r[q]);", "displacement(c, hub, s[q], r[q]);"),
    ("zero volume counted as positive",
     "odd[idx] += (v > 0) - (v < 0);", "odd[idx] += (v >= 0) - (v < 0);"),
    ("one spoke-spoke side not tested",
     "                if (pair_bin(&q->c, q->nbr[b], q->nbr[d]) < 0) continue;\n", ""),
    # six-bin 4pCF (§II.2, §III.2, §V.2)
    ("largest tuple taken as canonical",
     "        if (c < 0) {\n            memcpy(best, t, sizeof(t));", "        if (c > 0) {\n            memcpy(best, t, sizeof(t));"),
    ("every relabelling counted as even",
     "g_perm_par[c] = inv & 1;", "g_perm_par[c] = 0;"),
    ("tetrahedron volume from the wrong origin",
     "displacement(c, q[ord[0]], q[ord[k + 1]], r[k]);", "displacement(c, q[0], q[ord[k + 1]], r[k]);"),
    # weights (§II.1, §III.3)
    ("pairs weighted twice",
     "        for (int64_t j = i + 1; j < n; ++j) {\n            int b = pair_bin(&c, i, j);",
     "        for (int64_t j = 0; j < n; ++j) {\n            int b = pair_bin(&c, i, j);"),
    ("third weight of a triangle dropped",
     "+= (__int128)t->w[i] * t->w[j] * t->w[k];", "+= (__int128)t->w[i] * t->w[j];"),
    ("odd weighted sum without its sign",
     "od[idx] += sg * W;", "od[idx] += W;"),
]


def _build(src_text, workdir):
    src = os.path.join(workdir, "gs_oracle.c")
    lib = os.path.join(workdir, "liboracle.so")
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", lib, src],
                   check=True, capture_output=True)
    return src, lib


def _run_pins(src, lib):
    env = dict(os.environ, GS_ORACLE_SRC=src, GS_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", *PINS, "-x", "-q", "-m", "not gpu", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-2000:]


def test_unchanged_oracle_passes_through_the_same_harness(tmp_path):
    src, lib = _build(open(SRC).read(), str(tmp_path))
    rc, out = _run_pins(src, lib)
    assert rc == 0, out


def test_every_planted_mistake_fails_a_pin(tmp_path):
    original = open(SRC).read()
    jobs = []
    for k, (name, old, new) in enumerate(MUTANTS):
        assert original.count(old) == 1, f"mutation site of '{name}' not found exactly once"
        d = tmp_path / f"m{k}"
        d.mkdir()
        jobs.append((name, *_build(original.replace(old, new), str(d))))
    with ThreadPoolExecutor(max_workers=4) as pool:
        results = list(pool.map(lambda j: (j[0], *_run_pins(j[1], j[2])), jobs))
    survivors = [name for name, rc, _ in results if rc == 0]
    assert not survivors, f"planted mistakes no pin catches: {survivors}"
    # a caught mistake fails a pin; it neither crashes nor breaks collection
    odd = [(name, rc, out[-300:]) for name, rc, out in results if rc != 1]
    assert not odd, odd
