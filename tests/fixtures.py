"""Readers for the hand-derived fixtures in tests/golden/, and small helpers
shared by the tests (configuration enumeration, an independent NumPy brute
force used only to cross-check the oracle's loops on tiny inputs)."""
from __future__ import annotations

import itertools
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if line:
                yield line.split()


def pair_bin_cases():
    for t in _lines("pair_bins.txt"):
        box, periodic = int(t[0]), int(t[1])
        edges = [int(v) for v in t[2].split(",")]
        p = [int(v) for v in t[3:6]]
        q = [int(v) for v in t[6:9]]
        yield box, periodic, edges, p, q, int(t[9])


def triangle_fixtures():
    cur = None
    for t in _lines("triangles.txt"):
        if t[0] == "fixture":
            cur = {"name": t[1], "box": int(t[2]), "periodic": int(t[3]),
                   "edges": [int(v) for v in t[4].split(",")], "points": [], "expect": {}}
        elif t[0] == "point":
            cur["points"].append([int(v) for v in t[1:4]])
        elif t[0] == "expect":
            cur["expect"][tuple(int(v) for v in t[1:4])] = int(t[4])
        elif t[0] == "end":
            cur["points"] = np.array(cur["points"], dtype=np.int32)
            yield cur
            cur = None


def tetrahedron_shapes():
    cur = None
    for t in _lines("tetrahedra.txt"):
        if t[0] == "shape":
            cur = {"name": t[1], "vertices": [], "hubs": []}
        elif t[0] == "vertex":
            cur["vertices"].append([int(v) for v in t[1:4]])
        elif t[0] == "hub":
            cur["hubs"].append((int(t[1]), (int(t[2]), int(t[3]), int(t[4])), int(t[5]), int(t[6])))
        elif t[0] == "end":
            cur["vertices"] = np.array(cur["vertices"], dtype=np.int64)
            yield cur
            cur = None


TETRA_EDGES = [0, 1000, 2000, 3000, 4000]


def configs3(nb):
    """Sorted triples b1 <= b2 <= b3 in lexicographic order."""
    return [c for c in itertools.product(range(nb), repeat=3) if c[0] <= c[1] <= c[2]]


def configs4(nb):
    """Strictly increasing triples b1 < b2 < b3 in lexicographic order."""
    return [c for c in itertools.product(range(nb), repeat=3) if c[0] < c[1] < c[2]]


def np_bins(xyz, box, periodic, edges):
    """Bin matrix B[i, j] (-1 = no edge) and displacements d[i, j] = x_j - x_i."""
    x = np.asarray(xyz, dtype=np.int64)
    d = x[None, :, :] - x[:, None, :]
    if periodic:
        d = np.where(2 * d >= box, d - box, d)
        d = np.where(2 * d < -box, d + box, d)
    d2 = np.einsum("ijk,ijk->ij", d, d)
    e2 = np.asarray(edges, dtype=np.int64) ** 2
    b = np.searchsorted(e2, d2, side="right") - 1
    ok = (d2 >= e2[0]) & (d2 < e2[-1])
    np.fill_diagonal(ok, False)
    return np.where(ok, b, -1), d


def np_brute3(xyz, box, periodic, edges):
    nb = len(edges) - 1
    B, _ = np_bins(xyz, box, periodic, edges)
    index = {c: n for n, c in enumerate(configs3(nb))}
    hist = np.zeros(len(index), dtype=np.uint64)
    n = len(xyz)
    if n < 3:
        return hist
    tri = np.array(list(itertools.combinations(range(n), 3)), dtype=np.int64)
    bij, bik, bjk = B[tri[:, 0], tri[:, 1]], B[tri[:, 0], tri[:, 2]], B[tri[:, 1], tri[:, 2]]
    ok = (bij >= 0) & (bik >= 0) & (bjk >= 0)
    s = np.sort(np.stack([bij, bik, bjk], axis=1)[ok], axis=1)
    for row in s:
        hist[index[tuple(int(v) for v in row)]] += 1
    return hist


def det3(r1, r2, r3):
    """Determinant of the rows r1, r2, r3 by cofactor expansion along r1 (Python ints)."""
    a, b, c = (int(v) for v in r1)
    d, e, f = (int(v) for v in r2)
    g, h, i = (int(v) for v in r3)
    return a * (e * i - f * h) - b * (d * i - f * g) + c * (d * h - e * g)


def np_brute4(xyz, box, periodic, edges):
    nb = len(edges) - 1
    B, D = np_bins(xyz, box, periodic, edges)
    index = {c: n for n, c in enumerate(configs4(nb))}
    even = np.zeros(len(index), dtype=np.uint64)
    odd = np.zeros(len(index), dtype=np.int64)
    n = len(xyz)
    for i in range(n):
        spokes = [j for j in range(n) if B[i, j] >= 0]
        for j, k, l in itertools.combinations(spokes, 3):
            if B[j, k] < 0 or B[j, l] < 0 or B[k, l] < 0:
                continue
            trio = sorted([(B[i, j], j), (B[i, k], k), (B[i, l], l)])
            bins = tuple(int(t[0]) for t in trio)
            if len(set(bins)) < 3:
                continue
            v = det3(D[i, trio[0][1]], D[i, trio[1][1]], D[i, trio[2][1]])
            even[index[bins]] += 1
            odd[index[bins]] += (v > 0) - (v < 0)
    return even, odd
