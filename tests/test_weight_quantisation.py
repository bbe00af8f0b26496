"""The error of int16 fixed-point weights against real (FP64) weights.

The paper accumulates signed FP64 weights (GRAMSCI v2 §II.1); this library
takes int16 fixed-point weights so that every weighted sum is an exact
integer. A real weight w with |w| <= 1 becomes q = round(S w), S = 32767
(quantize_weights), i.e. w~ = q / S with |w~ - w| <= 1 / (2 S) and |w~| <= 1.
A pair, triangle or tetrahedron term is the product of k vertex weights
(k = 2, 3, 4), and for factors of modulus at most 1 the telescoping sum
  prod w~ - prod w = sum_v (w~_v - w_v) prod_{u<v} w_u prod_{u>v} w~_u
gives |prod w~ - prod w| <= k / (2 S) exactly (no higher-order terms). So a
configuration summing n terms is within n k / (2 S) of the FP64 sum, before
the FP64 sum's own rounding. These tests check that bound with the oracle's
exact integer sums (divided by S^k) against FP64 brute-force sums of the
unquantised weights, for signed data-minus-random style weights and for
positive FKP-like weights, and check that the bound is attained to within
a modest factor by adversarial weights (so it is not loose)."""
import itertools
import math

import numpy as np
import pytest

import oracle
from cosmology_point_correlation_gb300 import catalogues, quantize_weights, WEIGHT_SCALE


def _pairs_and_triangles(xyz, box, edges):
    g = oracle.graph(xyz, box, 1, edges)
    n = len(xyz)
    adj = [dict(zip(g.nbr[g.row_ptr[i]:g.row_ptr[i + 1]], g.bin[g.row_ptr[i]:g.row_ptr[i + 1]])) for i in range(n)]
    pairs = [(i, j, b) for i in range(n) for j, b in adj[i].items() if j > i]
    tris = []
    for i in range(n):
        fw = sorted(j for j in adj[i] if j > i)
        for a, j in enumerate(fw):
            for k in fw[a + 1:]:
                if k in adj[j]:
                    tris.append((i, j, k, tuple(sorted((adj[i][j], adj[i][k], adj[j][k])))))
    return pairs, tris


@pytest.mark.parametrize("kind", ["signed", "fkp"])
def test_quantised_weights_stay_within_the_bound(kind):
    box = catalogues.box_lattice(40.0)
    xyz = catalogues.neyman_scott(350, 40.0, 12, 30.0, 2.0, 5)
    edges = catalogues.linear_edges_lu(8.0, 4)
    nb = len(edges) - 1
    rng = np.random.default_rng(11)
    if kind == "signed":      # data +1/N_D-like and random -1/N_R-like weights, rescaled to |w| <= 1
        w = np.where(rng.uniform(size=len(xyz)) < 0.5, 1.0, -0.73) * rng.uniform(0.2, 1.0, len(xyz))
    else:                      # FKP-like 1 / (1 + n P) in (0, 1]
        w = 1.0 / (1.0 + rng.lognormal(0.0, 1.0, len(xyz)))
    q = quantize_weights(w)
    assert q.dtype == np.int16 and np.all(np.abs(q.astype(np.int64) / WEIGHT_SCALE - w) <= 0.5 / WEIGHT_SCALE)
    pairs, tris = _pairs_and_triangles(xyz, box, edges)
    S = WEIGHT_SCALE

    exact2 = oracle.count_2pcf_weighted(xyz, box, 1, edges, q)
    f2 = np.zeros(nb)
    n2 = np.zeros(nb, dtype=np.int64)
    for i, j, b in pairs:
        f2[b] += w[i] * w[j]
        n2[b] += 1
    for b in range(nb):
        err = abs(exact2[b] / S ** 2 - f2[b])
        assert err <= n2[b] * 2 / (2 * S) + 1e-12 * max(1.0, abs(f2[b]))

    cfg = {c: k for k, c in enumerate(c for c in itertools.combinations_with_replacement(range(nb), 3))}
    exact3 = oracle.count_3pcf_weighted(xyz, box, 1, edges, q)
    f3 = np.zeros(len(cfg))
    n3 = np.zeros(len(cfg), dtype=np.int64)
    for i, j, k, c in tris:
        f3[cfg[c]] += w[i] * w[j] * w[k]
        n3[cfg[c]] += 1
    assert n3.sum() > 1000
    for c in range(len(cfg)):
        err = abs(exact3[c] / S ** 3 - f3[c])
        assert err <= n3[c] * 3 / (2 * S) + 1e-12 * max(1.0, abs(f3[c]))


def test_the_bound_is_attained_by_adversarial_weights():
    # every weight sits half a step below a representable value, all of one
    # sign: each factor's error is 1/(2S) - tiny in the same direction, so a
    # pair's error is close to 2/(2S) (the bound, up to the factors' moduli)
    S = WEIGHT_SCALE
    w = np.full(6, (S - 0.5 + 1e-9) / S)
    q = quantize_weights(w)
    err = abs((int(q[0]) / S) * (int(q[1]) / S) - w[0] * w[1])
    assert 0.9 * 2 / (2 * S) <= err <= 2 / (2 * S)


def test_quantize_rejects_weights_outside_the_unit_interval():
    with pytest.raises(ValueError):
        quantize_weights(np.array([0.5, 1.0001]))
    assert quantize_weights(np.array([1.0, -1.0, 0.0])).tolist() == [32767, -32767, 0]
    assert math.isclose(WEIGHT_SCALE, 32767)
