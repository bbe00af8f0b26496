"""Pins of the oracle's six-edge-bin 4pCF (GRAMSCI v2 §II.2 tetrahedra, §III.2
Eq.(3) handedness, §V.2: 276 tetrahedron configurations for 4 radial bins).

Configuration of a tetrahedron: the lexicographically smallest
(b01, b02, b03, b12, b13, b23) over the 24 orderings of its vertices;
configurations numbered in lexicographic order of those tuples. Odd channel:
sign of V = det[x1 - x0; x2 - x0; x3 - x0] for an ordering reaching the smallest
tuple, 0 when orderings of both parities reach it (achiral) or V = 0.
"""
import itertools

import numpy as np
import pytest

import oracle
from cosmology_point_correlation_gb300 import catalogues
from tests import fixtures as fx

PAIRS = [(0, 1), (0, 2), (0, 3), (1, 2), (1, 3), (2, 3)]


def _canon(bm):
    """Independent canonical form: (tuple, chiral, one minimal ordering)."""
    best, par, order = None, set(), None
    for p in itertools.permutations(range(4)):
        t = tuple(bm[p[a]][p[b]] for a, b in PAIRS)
        inv = sum(p[x] > p[y] for x in range(4) for y in range(x + 1, 4)) & 1
        if best is None or t < best:
            best, par, order = t, {inv}, p
        elif t == best:
            par.add(inv)
    return best, len(par) == 1, order


def _canonical_list(nb):
    out = []
    for t in itertools.product(range(nb), repeat=6):
        bm = [[0] * 4 for _ in range(4)]
        for (a, b), v in zip(PAIRS, t):
            bm[a][b] = bm[b][a] = v
        if _canon(bm)[0] == t:
            out.append(t)
    return out


def test_configuration_count_matches_paper_and_burnside():
    assert oracle.nconfig6(4) == 276                      # §V.2: 276 configurations, 4 bins
    for nb in range(1, 7):
        assert oracle.nconfig6(nb) == (nb ** 6 + 9 * nb ** 4 + 14 * nb ** 2) // 24


def test_configuration_index_is_lexicographic_rank():
    cl = _canonical_list(3)
    assert len(cl) == oracle.nconfig6(3)
    for k, t in enumerate(cl):
        assert oracle.config_index6(3, t) == k
    assert oracle.config_index6(3, (1, 0, 0, 0, 0, 0)) == -1


def _np_brute_six(xyz, box, periodic, edges):
    nb = len(edges) - 1
    B, D = fx.np_bins(xyz, box, periodic, edges)
    index = {t: k for k, t in enumerate(_canonical_list(nb))}
    even = np.zeros(len(index), dtype=np.uint64)
    odd = np.zeros(len(index), dtype=np.int64)
    for q in itertools.combinations(range(len(xyz)), 4):
        bm = [[B[q[a], q[b]] if a != b else 0 for b in range(4)] for a in range(4)]
        if min(bm[a][b] for a, b in PAIRS) < 0:
            continue
        t, chiral, o = _canon(bm)
        even[index[t]] += 1
        if chiral:
            v = fx.det3(D[q[o[0]], q[o[1]]], D[q[o[0]], q[o[2]]], D[q[o[0]], q[o[3]]])
            odd[index[t]] += (v > 0) - (v < 0)
    return even, odd


@pytest.mark.parametrize("periodic", [0, 1])
@pytest.mark.parametrize("seed", [3, 4])
def test_matches_independent_brute_force(periodic, seed):
    box = 9000
    xyz = catalogues.neyman_scott(34, box / 1024, 3, 12.0, 1.2, seed)
    edges = [0, 1300, 2600, 4400]
    ref_e, ref_o = _np_brute_six(xyz, box, periodic, edges)
    assert ref_e.sum() > 20 and np.abs(ref_o).sum() > 0
    for fn in (oracle.brute4six, oracle.count_4pcf6):
        e, o = fn(xyz, box, periodic, edges)
        assert np.array_equal(e, ref_e) and np.array_equal(o, ref_o)


def test_hand_derived_tetrahedra():
    # edges 0,1000,...,4000 (4 bins). T: bins AB 0, AC 1, AD 2, BC 2, BD 2, CD 3;
    # the smallest tuple starts with the only bin-0 pair AB, then AC (bin 1):
    # ordering (A, B, C, D) -> (0,1,2,2,2,3), reached by no other ordering
    # (chiral); V = det[B-A; C-A; D-A] = 700*1900*2500 > 0 -> odd +1, mirror -1.
    # R (regular): all bins 1 -> (1,1,1,1,1,1), reached by all 24 orderings
    # (achiral): even 1, odd 0. P (coplanar): V = 0 -> odd 0.
    shapes = {s["name"]: s for s in fx.tetrahedron_shapes()}
    edges = fx.TETRA_EDGES
    box = 1_000_000
    k_t = oracle.config_index6(4, (0, 1, 2, 2, 2, 3))
    k_r = oracle.config_index6(4, (1, 1, 1, 1, 1, 1))
    expect = {"T": {k_t: (1, 1)}, "T_relabel": {k_t: (1, 1)}, "T_mirror": {k_t: (1, -1)},
              "R": {k_r: (1, 0)}}
    for name, want in expect.items():
        xyz = (shapes[name]["vertices"] + 50_000).astype(np.int32)
        e, o = oracle.count_4pcf6(xyz, box, 0, edges)
        got = {k: (int(e[k]), int(o[k])) for k in np.nonzero(e)[0]}
        assert got == want, name
    xyz = (shapes["P"]["vertices"] + 50_000).astype(np.int32)
    e, o = oracle.count_4pcf6(xyz, box, 0, edges)
    assert e.sum() == 1 and not o.any()


@pytest.mark.parametrize("periodic", [0, 1])
def test_invariances_and_hub_ranges(periodic):
    box = 20000
    xyz = catalogues.neyman_scott(300, box / 1024, 6, 50.0, 1.5, 12)
    edges = catalogues.linear_edges_lu(4.0, 4)
    g = oracle.graph(xyz, box, periodic, edges)
    e, o = oracle.count_4pcf6(xyz, box, periodic, edges, g)
    assert e.sum() > 1000 and np.abs(o).sum() > 0
    perm = np.random.default_rng(0).permutation(len(xyz))
    e2, o2 = oracle.count_4pcf6(xyz[perm], box, periodic, edges)
    assert np.array_equal(e2, e) and np.array_equal(o2, o)
    m = xyz.astype(np.int64).copy()
    m[:, 0] = (box - m[:, 0]) % box if periodic else box - 1 - m[:, 0]
    e3, o3 = oracle.count_4pcf6(m.astype(np.int32), box, periodic, edges)
    assert np.array_equal(e3, e) and np.array_equal(o3, -o)
    parts = [oracle.count_4pcf6(xyz, box, periodic, edges, g, a, b) for a, b in [(0, 77), (77, 300)]]
    assert np.array_equal(parts[0][0] + parts[1][0], e) and np.array_equal(parts[0][1] + parts[1][1], o)


# ---------------------------------------------------------------- weighted (§II.1 signed weights)

def _np_brute_six_weighted(xyz, box, periodic, edges, w):
    """Python big-int sums of w_a w_b w_c w_d (even) and sign x that (odd)."""
    nb = len(edges) - 1
    B, D = fx.np_bins(xyz, box, periodic, edges)
    index = {t: k for k, t in enumerate(_canonical_list(nb))}
    even = [0] * len(index)
    odd = [0] * len(index)
    for q in itertools.combinations(range(len(xyz)), 4):
        bm = [[B[q[a], q[b]] if a != b else 0 for b in range(4)] for a in range(4)]
        if min(bm[a][b] for a, b in PAIRS) < 0:
            continue
        t, chiral, o = _canon(bm)
        W = int(w[q[0]]) * int(w[q[1]]) * int(w[q[2]]) * int(w[q[3]])
        even[index[t]] += W
        if chiral:
            v = fx.det3(D[q[o[0]], q[o[1]]], D[q[o[0]], q[o[2]]], D[q[o[0]], q[o[3]]])
            odd[index[t]] += ((v > 0) - (v < 0)) * W
    return even, odd


@pytest.mark.parametrize("periodic", [0, 1])
def test_weighted_matches_big_int_brute_force(periodic):
    box = 9000
    xyz = catalogues.neyman_scott(34, box / 1024, 3, 12.0, 1.2, 5 + periodic)
    edges = [0, 1300, 2600, 4400]
    w = np.random.default_rng(9 + periodic).integers(-32767, 32768, size=len(xyz)).astype(np.int16)
    ref_e, ref_o = _np_brute_six_weighted(xyz, box, periodic, edges, w)
    assert sum(1 for v in ref_e if v) > 3 and any(ref_o)
    assert oracle.count_4pcf6_weighted(xyz, box, periodic, edges, w) == (ref_e, ref_o)


def test_weighted_reduces_to_counts_and_subcatalogues():
    box = 20000
    xyz = catalogues.neyman_scott(300, box / 1024, 6, 50.0, 1.5, 12)
    edges = catalogues.linear_edges_lu(4.0, 4)
    e, o = oracle.count_4pcf6(xyz, box, 1, edges)
    assert e.sum() > 1000
    one = np.ones(len(xyz), np.int16)
    assert oracle.count_4pcf6_weighted(xyz, box, 1, edges, one) == ([int(v) for v in e], [int(v) for v in o])
    # a constant weight c scales both channels by c^4 (here beyond 2^63)
    c = -32767
    we, wo = oracle.count_4pcf6_weighted(xyz, box, 1, edges, np.full(len(xyz), c, np.int16))
    assert we == [int(v) * c ** 4 for v in e] and wo == [int(v) * c ** 4 for v in o]
    assert max(we) > 1 << 63
    # 0/1 weights: only tetrahedra with all four vertices in the subset count,
    # which is the unweighted count of the subset alone
    keep = np.random.default_rng(1).uniform(size=len(xyz)) < 0.7
    se, so = oracle.count_4pcf6(xyz[keep], box, 1, edges)
    assert oracle.count_4pcf6_weighted(xyz, box, 1, edges, keep.astype(np.int16)) == \
        ([int(v) for v in se], [int(v) for v in so])
    # hub ranges add up
    w = np.random.default_rng(2).integers(-32767, 32768, size=len(xyz)).astype(np.int16)
    g = oracle.graph(xyz, box, 1, edges)
    full = oracle.count_4pcf6_weighted(xyz, box, 1, edges, w, g)
    p1 = oracle.count_4pcf6_weighted(xyz, box, 1, edges, w, g, 0, 123)
    p2 = oracle.count_4pcf6_weighted(xyz, box, 1, edges, w, g, 123, 300)
    assert [x + y for x, y in zip(p1[0], p2[0])] == full[0]
    assert [x + y for x, y in zip(p1[1], p2[1])] == full[1]
