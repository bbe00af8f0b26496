"""Closed-form pins of the oracle on uniform (Poisson-like) catalogues. CPU only.

For N iid uniform points on a periodic cube of side L (lattice units):

* pairs: a pair is in bin b with probability p_b = (4 pi / 3)(e_{b+1}^3 - e_b^3) / L^3,
  and on the torus the C(N,2) pair indicators are pairwise independent, so the
  count has mean C(N,2) p_b and variance C(N,2) p_b (1 - p_b).
* triangles: fixing x1, the sides r1 = |x2 - x1| and r2 = |x3 - x1| have
  densities 4 pi r^2 / L^3 and the angle between them has uniform cosine, so
  (r1, r2, r3) has joint density 8 pi^2 r1 r2 r3 / L^6 on the region obeying the
  triangle inequality. The expected count in the sorted configuration
  (b1 <= b2 <= b3) is C(N,3) 8 pi^2 / L^6 times the sum, over the distinct
  orderings (s1, s2, s3) of (b1, b2, b3), of the integral of r1 r2 r3 over
  s1 x s2 x s3 under the triangle inequality. Summed over all configurations
  this is C(N,3) p^2 15/32 with p = (4 pi / 3) R^3 / L^3 (15/32 being the
  chance that two uniform points in a ball of radius R are closer than R).
* parity: a uniform catalogue is statistically mirror symmetric, so the odd
  channel averages to zero (the GRAMSCI v2 paper's parity null, §IV.9).

Triangle counts are correlated, so their scatter is taken from the ensemble.
"""
import itertools
import math

import numpy as np
import pytest

import oracle
from cosmology_point_correlation_gb300 import catalogues, configs
from tests import fixtures as fx


def _shell_integral(a1, b1, a2, b2, a3, b3, m=400):
    """Integral of r1 r2 r3 over [a1,b1] x [a2,b2] x [a3,b3] where the three
    sides obey the triangle inequality; exact in r3, midpoint rule in r1, r2."""
    r1 = a1 + (np.arange(m) + 0.5) * (b1 - a1) / m
    r2 = a2 + (np.arange(m) + 0.5) * (b2 - a2) / m
    R1, R2 = np.meshgrid(r1, r2, indexing="ij")
    lo = np.maximum(a3, np.abs(R1 - R2))
    hi = np.minimum(b3, R1 + R2)
    g = np.where(hi > lo, 0.5 * (hi * hi - lo * lo), 0.0)
    return float((R1 * R2 * g).sum() * (b1 - a1) * (b2 - a2) / (m * m))


def expected_triangles(n, box, edges):
    nb = len(edges) - 1
    e = np.asarray(edges, dtype=np.float64) / box          # in units of the box side
    I = np.zeros((nb, nb, nb))
    for s1, s2, s3 in itertools.product(range(nb), repeat=3):
        I[s1, s2, s3] = _shell_integral(e[s1], e[s1 + 1], e[s2], e[s2 + 1], e[s3], e[s3 + 1])
    out = []
    for c in fx.configs3(nb):
        out.append(sum(I[p] for p in set(itertools.permutations(c))))
    return math.comb(n, 3) * 8 * math.pi ** 2 * np.array(out)


def test_triangle_integral_total():
    # the per-configuration integrals must add up to the closed-form total
    w = configs.TINY_3PCF
    e = expected_triangles(w.n, w.box_lu, w.edges_lu)
    p = 4 * math.pi / 3 * (w.edges_lu[-1] / w.box_lu) ** 3
    total = math.comb(w.n, 3) * p * p * 15 / 32
    assert abs(e.sum() / total - 1) < 2e-4
    assert abs(total - 7.006e5) / 7.006e5 < 1e-3


@pytest.fixture(scope="module")
def tiny_ensemble():
    w = configs.TINY_3PCF
    pairs, tris = [], []
    for seed in range(2000, 2032):
        xyz = w.points(seed=seed)
        g = oracle.graph(xyz, w.box_lu, 1, w.edges_lu)
        pairs.append(oracle.count_2pcf(xyz, w.box_lu, 1, w.edges_lu, g))
        tris.append(oracle.count_3pcf(xyz, w.box_lu, 1, w.edges_lu, g))
    return np.array(pairs, dtype=np.float64), np.array(tris, dtype=np.float64)


def test_pair_counts_closed_form(tiny_ensemble):
    w = configs.TINY_3PCF
    pairs, _ = tiny_ensemble
    e = w.edges_lu.astype(np.float64)
    p = 4 * math.pi / 3 * (e[1:] ** 3 - e[:-1] ** 3) / float(w.box_lu) ** 3
    mean = math.comb(w.n, 2) * p
    s = pairs.sum(axis=0)
    k = len(pairs)
    z = (s - k * mean) / np.sqrt(k * mean * (1 - p))
    assert np.all(np.abs(z) < 5), z


def test_triangle_counts_closed_form(tiny_ensemble):
    w = configs.TINY_3PCF
    _, tris = tiny_ensemble
    expect = expected_triangles(w.n, w.box_lu, w.edges_lu)
    mean = tris.mean(axis=0)
    sem = tris.std(axis=0, ddof=1) / math.sqrt(len(tris))
    use = expect >= 20
    assert use.sum() > 140
    z = (mean[use] - expect[use]) / sem[use]
    assert np.all(np.abs(z) < 5), np.sort(np.abs(z))[-5:]
    tot = tris.sum(axis=1)
    z_tot = (tot.mean() - expect.sum()) / (tot.std(ddof=1) / math.sqrt(len(tot)))
    assert abs(z_tot) < 5


def test_parity_odd_channel_null_on_uniform():
    box = 100 * 1024
    edges = np.arange(7, dtype=np.int64) * 2048
    evs, ods = [], []
    for seed in range(3000, 3012):
        xyz = catalogues.uniform(3000, 100.0, seed)
        ev, od = oracle.count_4pcf_parity(xyz, box, 1, edges)
        evs.append(ev)
        ods.append(od)
    ev = np.sum(evs, axis=0).astype(np.float64)
    od = np.sum(ods, axis=0).astype(np.float64)
    assert ev.sum() > 1e5
    # each tetrahedron is seen from up to four hubs, so allow a factor 2 in the scatter
    assert np.all(np.abs(od) <= 5 * 2 * np.sqrt(ev) + 5)
