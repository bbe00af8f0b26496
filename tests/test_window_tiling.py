"""The tile rules of the out-of-core mode (GRAMSCI v2 §III.5.3), checked on the
CPU against the oracle, independently of the CUDA code:

* 3pCF: tile (h, w) with w >= h counts the triangles (i < j < k) whose hub i
  lies in window h and whose spoke j lies in window w;
* parity 4pCF: tile (h, c1, c2) with c1 <= c2 counts, at hub i in window h,
  the cliques (s1 < s2 < s3 by position in the hub row) whose s1 lies in c1
  and s2 in c2.

Windows are contiguous index ranges cut at random; the tiles must add up to
the full histograms exactly, so that every triangle and clique falls in one
tile only."""
import itertools

import numpy as np
import pytest

import oracle
from cosmology_point_correlation_gb300 import catalogues
from tests import fixtures as fx


def _rows(g):
    return [g.nbr[g.row_ptr[i]:g.row_ptr[i + 1]] for i in range(len(g.row_ptr) - 1)]


def _windows(n, cuts, seed):
    rng = np.random.default_rng(seed)
    bounds = np.unique(np.concatenate([[0, n], rng.integers(1, n, size=cuts)]))
    win = np.zeros(n, dtype=np.int64)
    for w, (a, b) in enumerate(zip(bounds[:-1], bounds[1:])):
        win[a:b] = w
    return win, len(bounds) - 1


def _triangles(xyz, box, periodic, edges, g):
    """(i, j, k, configuration) of every triangle, i < j < k, from the rows."""
    rows = _rows(g)
    B, _ = fx.np_bins(xyz, box, periodic, edges)
    cfg = {t: k for k, t in enumerate(fx.configs3(len(edges) - 1))}
    out = []
    for i, row in enumerate(rows):
        fwd = [j for j in row if j > i]
        for a, j in enumerate(fwd):
            nj = set(rows[j])
            out += [(i, j, k, cfg[tuple(sorted((B[i, j], B[i, k], B[j, k])))]) for k in fwd[a + 1:] if k in nj]
    return np.array(out, dtype=np.int64).reshape(-1, 4)


def _cliques(xyz, box, periodic, edges, g):
    """(hub, s1, s2, configuration, odd sign) of every hub and spoke triple
    s1 < s2 < s3 (row positions) that is a clique with distinct hub bins."""
    rows = _rows(g)
    B, D = fx.np_bins(xyz, box, periodic, edges)
    cfg = {t: k for k, t in enumerate(fx.configs4(len(edges) - 1))}
    out = []
    for i, row in enumerate(rows):
        adj = [set(rows[j]) for j in row]
        for p1, p2, p3 in itertools.combinations(range(len(row)), 3):
            j1, j2, j3 = row[p1], row[p2], row[p3]
            if j2 not in adj[p1] or j3 not in adj[p1] or j3 not in adj[p2]:
                continue
            bins = (B[i, j1], B[i, j2], B[i, j3])
            if len(set(bins)) < 3:
                continue
            js = [(j1, j2, j3)[o] for o in np.argsort(bins)]
            v = fx.det3(D[i, js[0]], D[i, js[1]], D[i, js[2]])
            out.append((i, j1, j2, cfg[tuple(sorted(bins))], (v > 0) - (v < 0)))
    return np.array(out, dtype=np.int64).reshape(-1, 5)


@pytest.mark.parametrize("periodic,cuts,seed", [(0, 3, 1), (1, 5, 2), (1, 40, 3)])
def test_triangle_tiles_add_up(periodic, cuts, seed):
    box = 30000
    xyz = catalogues.neyman_scott(250, box / 1024, 8, 30.0, 2.0, 10 + seed)
    edges = [0, 2000, 4000, 6000]
    g = oracle.graph(xyz, box, periodic, edges)
    t = _triangles(xyz, box, periodic, edges, g)
    win, nw = _windows(len(xyz), cuts, seed)
    hist = np.zeros(len(fx.configs3(3)), dtype=np.int64)
    seen = np.zeros(len(t), dtype=np.int64)
    for h in range(nw):
        for w in range(h, nw):
            m = (win[t[:, 0]] == h) & (win[t[:, 1]] == w)
            np.add.at(hist, t[m, 3], 1)
            seen += m
    assert len(t) > 100 and np.all(seen == 1)               # every triangle in exactly one tile
    assert np.array_equal(hist, oracle.count_3pcf(xyz, box, periodic, edges, g).astype(np.int64))


@pytest.mark.parametrize("periodic,cuts,seed", [(0, 3, 4), (1, 7, 5), (1, 30, 6)])
def test_clique_tiles_add_up(periodic, cuts, seed):
    box = 30000
    xyz = catalogues.neyman_scott(160, box / 1024, 6, 25.0, 2.0, 20 + seed)
    edges = [0, 1500, 3000, 4500, 6000]
    g = oracle.graph(xyz, box, periodic, edges)
    c = _cliques(xyz, box, periodic, edges, g)
    win, nw = _windows(len(xyz), cuts, seed)
    even = np.zeros(len(fx.configs4(4)), dtype=np.int64)
    odd = np.zeros_like(even)
    seen = np.zeros(len(c), dtype=np.int64)
    for h in range(nw):
        for c1, c2 in itertools.combinations_with_replacement(range(nw), 2):
            m = (win[c[:, 0]] == h) & (win[c[:, 1]] == c1) & (win[c[:, 2]] == c2)
            np.add.at(even, c[m, 3], 1)
            np.add.at(odd, c[m, 3], c[m, 4])
            seen += m
    ref_e, ref_o = oracle.count_4pcf_parity(xyz, box, periodic, edges, g)
    assert len(c) > 50 and np.all(seen == 1)               # every clique in exactly one tile
    assert np.array_equal(even, ref_e.astype(np.int64)) and np.array_equal(odd, ref_o)
