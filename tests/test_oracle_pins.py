"""Pins for the CPU oracle: hand-derived fixtures, an independent brute force,
and exact invariants. CPU only.

Sources (GRAMSCI v2 paper, "Fast Graph-based Higher-Order Clustering
Statistics on the GPU"): §II.1 Eq.(1) (sorted neighbour lists with a bin byte),
§II.2 (hub-and-spoke triangles), §III.2 Eq.(3) (signed volume, degenerate
rule), §IV.9 (chiral injection: left +1, right -1 in the odd count),
§V.1 Fig.8 (220 configurations for 10 radial bins, lexicographic order).
"""
import itertools

import numpy as np
import pytest

import oracle
from cosmology_point_correlation_gb300 import catalogues
from tests import fixtures as fx


# ---------------------------------------------------------------- pair rule

@pytest.mark.parametrize("case", list(fx.pair_bin_cases()))
def test_pair_rule_fixture(case):
    box, periodic, edges, p, q, expect = case
    xyz = np.array([p, q], dtype=np.int32)
    nbr, bins = oracle.row(xyz, box, periodic, edges, 0)
    if expect < 0:
        assert len(nbr) == 0
    else:
        assert list(nbr) == [1] and list(bins) == [expect]
    # symmetric
    nbr2, bins2 = oracle.row(xyz, box, periodic, edges, 1)
    assert list(bins2) == list(bins)


def test_configuration_counts_match_paper():
    # §V.1 / Fig.8: 10 radial bins give 220 sorted triangle configurations.
    assert oracle.nconfig3(10) == 220
    for nb in range(1, 12):
        assert oracle.nconfig3(nb) == len(fx.configs3(nb))
        assert max(oracle.nconfig4(nb), 0) == len(fx.configs4(nb))


# ---------------------------------------------------------------- graph

@pytest.mark.parametrize("periodic", [0, 1])
@pytest.mark.parametrize("seed", [1, 2, 3])
def test_graph_matches_numpy_bins(periodic, seed):
    box = 20000
    xyz = catalogues.uniform(150, box / 1024, seed)
    edges = [0, 1000, 2500, 3000, 5000]
    g = oracle.graph(xyz, box, periodic, edges)
    B, _ = fx.np_bins(xyz, box, periodic, edges)
    for i in range(len(xyz)):
        r = slice(g.row_ptr[i], g.row_ptr[i + 1])
        js = np.nonzero(B[i] >= 0)[0]
        assert np.array_equal(g.nbr[r], js)
        assert np.array_equal(g.bin[r], B[i, js])


def test_graph_invariants():
    w = catalogues
    xyz = w.neyman_scott(600, 60.0, 12, 50.0, 2.0, 7)
    box = w.box_lattice(60.0)
    edges = w.linear_edges_lu(8.0, 6)
    g = oracle.graph(xyz, box, 1, edges)
    n = len(xyz)
    assert g.n_edges % 2 == 0
    adj = {}
    for i in range(n):
        row = g.nbr[g.row_ptr[i]:g.row_ptr[i + 1]]
        assert np.all(np.diff(row) > 0), "rows strictly increasing (Eq.1)"
        assert i not in set(row.tolist()), "no self loops"
        for j, b in zip(row, g.bin[g.row_ptr[i]:g.row_ptr[i + 1]]):
            adj[(i, int(j))] = int(b)
    for (i, j), b in adj.items():
        assert adj[(j, i)] == b, "symmetric adjacency with equal bins"


# ---------------------------------------------------------------- 3pCF

def _hist_dict(hist, nb):
    cfg = fx.configs3(nb)
    return {cfg[k]: int(v) for k, v in enumerate(hist) if v}


@pytest.mark.parametrize("fixture", list(fx.triangle_fixtures()), ids=lambda f: f["name"])
def test_3pcf_fixture(fixture):
    f = fixture
    nb = len(f["edges"]) - 1
    for fn in (oracle.count_3pcf, oracle.brute3):
        hist = fn(f["points"], f["box"], f["periodic"], f["edges"])
        assert _hist_dict(hist, nb) == f["expect"]
    assert _hist_dict(fx.np_brute3(f["points"], f["box"], f["periodic"], f["edges"]), nb) == f["expect"]


def test_3pcf_packed_index_is_lexicographic():
    # a single triangle with sorted bins (b1,b2,b3) lands at its rank in the
    # lexicographic list of sorted triples; sides along the axes of a right corner.
    nb = 5
    w = 1000
    edges = [k * w for k in range(nb + 1)]
    cfg = fx.configs3(nb)
    # right triangle with legs a, b: sides a, b, sqrt(a^2+b^2)
    for a, b in [(500, 500), (500, 1500), (1500, 2500), (2500, 3500), (500, 4900 // 2)]:
        xyz = np.array([[0, 0, 0], [a, 0, 0], [0, b, 0]], dtype=np.int32) + 10000
        hyp2 = a * a + b * b
        bins = sorted([a // w, b // w, int(np.searchsorted(np.array(edges) ** 2, hyp2, side="right") - 1)])
        if bins[2] >= nb:
            continue
        hist = oracle.count_3pcf(xyz, 100000, 0, edges)
        assert np.nonzero(hist)[0].tolist() == [cfg.index(tuple(bins))]


@pytest.mark.parametrize("periodic", [0, 1])
@pytest.mark.parametrize("seed", [11, 12, 13, 14])
def test_3pcf_matches_numpy_brute_force(periodic, seed):
    box = 16000
    xyz = catalogues.neyman_scott(110, box / 1024, 6, 15.0, 1.5, seed)
    edges = [0, 700, 1500, 2600, 4000]
    ref = fx.np_brute3(xyz, box, periodic, edges)
    assert ref.sum() > 50
    assert np.array_equal(oracle.count_3pcf(xyz, box, periodic, edges), ref)
    assert np.array_equal(oracle.brute3(xyz, box, periodic, edges), ref)


@pytest.mark.parametrize("periodic", [0, 1])
def test_3pcf_matches_brute3_larger(periodic):
    box = 40000
    xyz = catalogues.uniform(400, box / 1024, 99 + periodic)
    edges = catalogues.linear_edges_lu(9.0, 7)
    assert np.array_equal(oracle.count_3pcf(xyz, box, periodic, edges),
                          oracle.brute3(xyz, box, periodic, edges))


def test_3pcf_trace_invariant():
    # sum over undirected edges of |N(u) & N(v)| = 3 * number of triangles
    box = 30000
    xyz = catalogues.neyman_scott(500, box / 1024, 10, 50.0, 1.0, 5)
    edges = catalogues.linear_edges_lu(5.0, 5)
    g = oracle.graph(xyz, box, 1, edges)
    rows = [set(g.nbr[g.row_ptr[i]:g.row_ptr[i + 1]].tolist()) for i in range(len(xyz))]
    trace = sum(len(rows[u] & rows[v]) for u in range(len(xyz)) for v in rows[u] if v > u)
    hist = oracle.count_3pcf(xyz, box, 1, edges, g)
    assert trace == 3 * int(hist.sum()) and trace > 0


def test_3pcf_hub_ranges_sum_to_full():
    box = 30000
    xyz = catalogues.uniform(700, box / 1024, 21)
    edges = catalogues.linear_edges_lu(6.0, 4)
    g = oracle.graph(xyz, box, 1, edges)
    full = oracle.count_3pcf(xyz, box, 1, edges, g)
    cuts = [0, 1, 100, 333, 699, 700]
    parts = sum(oracle.count_3pcf(xyz, box, 1, edges, g, a, b) for a, b in zip(cuts, cuts[1:]))
    assert np.array_equal(parts, full)


def _mirror(xyz, box, periodic):
    m = xyz.astype(np.int64).copy()
    m[:, 0] = (box - m[:, 0]) % box if periodic else box - 1 - m[:, 0]
    return m.astype(np.int32)


@pytest.mark.parametrize("periodic", [0, 1])
def test_3pcf_geometric_invariances(periodic):
    box = 40000
    xyz = catalogues.neyman_scott(800, box / 1024, 16, 50.0, 1.5, 31)
    edges = catalogues.linear_edges_lu(6.0, 6)
    base = oracle.count_3pcf(xyz, box, periodic, edges)
    assert base.sum() > 1000
    rng = np.random.default_rng(0)
    perm = rng.permutation(len(xyz))
    assert np.array_equal(oracle.count_3pcf(xyz[perm], box, periodic, edges), base)
    assert np.array_equal(oracle.count_3pcf(_mirror(xyz, box, periodic), box, periodic, edges), base)
    assert np.array_equal(oracle.count_3pcf(np.ascontiguousarray(xyz[:, [1, 2, 0]]), box, periodic, edges), base)
    if periodic:
        t = np.array([12345, 777, 39999], dtype=np.int64)
        moved = ((xyz.astype(np.int64) + t) % box).astype(np.int32)
        assert np.array_equal(oracle.count_3pcf(moved, box, periodic, edges), base)


# ---------------------------------------------------------------- parity 4pCF

def _place(shapes_and_origins, box):
    pts = []
    for verts, origin in shapes_and_origins:
        pts.extend(((verts + np.asarray(origin)) % box).tolist())
    return np.array(pts, dtype=np.int32)


@pytest.mark.parametrize("periodic", [0, 1])
@pytest.mark.parametrize("shape", list(fx.tetrahedron_shapes()), ids=lambda s: s["name"])
def test_4pcf_fixture_per_hub(shape, periodic):
    box = 100000
    # periodic: straddle the corner of the box so every axis wraps
    origin = (99000, 99500, 98000) if periodic else (50000, 50000, 50000)
    xyz = _place([(shape["vertices"], origin)], box)
    edges = fx.TETRA_EDGES
    cfg = fx.configs4(len(edges) - 1)
    expect_even = np.zeros(len(cfg), dtype=np.uint64)
    expect_odd = np.zeros(len(cfg), dtype=np.int64)
    listed = {h[0]: h for h in shape["hubs"]}
    for v in range(4):
        ev, od = oracle.count_4pcf_parity_hubs(xyz, box, periodic, edges, [v])
        if v in listed:
            _, bins, e, o = listed[v]
            k = cfg.index(bins)
            assert np.nonzero(ev)[0].tolist() == [k] and ev[k] == e and od[k] == o
            assert np.count_nonzero(od) == (1 if o else 0)
            expect_even[k] += e
            expect_odd[k] += o
        else:
            assert not ev.any() and not od.any()
    for fn in (oracle.count_4pcf_parity, oracle.brute4):
        ev, od = fn(xyz, box, periodic, edges)
        assert np.array_equal(ev, expect_even) and np.array_equal(od, expect_odd)


def test_4pcf_chiral_injection_count_level():
    # §IV.9: n_L left and n_R right copies of one chiral unit, isolated from each
    # other, give odd = (n_L - n_R) * template and even = (n_L + n_R) * template.
    shapes = {s["name"]: s for s in fx.tetrahedron_shapes()}
    left, right = shapes["T"]["vertices"], shapes["T_mirror"]["vertices"]
    edges = fx.TETRA_EDGES
    box = 1_000_000
    ev1, od1 = oracle.count_4pcf_parity(_place([(left, (5000, 5000, 5000))], box), box, 0, edges)
    assert od1.any()
    for n_left, n_right in [(5, 0), (3, 2), (1, 4), (7, 7)]:
        placed = []
        for c in range(n_left + n_right):
            origin = (5000 + 12000 * (c % 8), 5000 + 12000 * (c // 8), 5000)
            placed.append((left if c < n_left else right, origin))
        xyz = _place(placed, box)
        ev, od = oracle.count_4pcf_parity(xyz, box, 0, edges)
        assert np.array_equal(ev, ev1 * np.uint64(n_left + n_right))
        assert np.array_equal(od, od1 * (n_left - n_right))


@pytest.mark.parametrize("periodic", [0, 1])
@pytest.mark.parametrize("seed", [41, 42, 43])
def test_4pcf_matches_numpy_brute_force(periodic, seed):
    box = 9000
    xyz = catalogues.neyman_scott(45, box / 1024, 3, 15.0, 1.2, seed)
    edges = [0, 900, 1700, 2600, 3300, 4400]
    ev_ref, od_ref = fx.np_brute4(xyz, box, periodic, edges)
    assert ev_ref.sum() > 20
    for fn in (oracle.count_4pcf_parity, oracle.brute4):
        ev, od = fn(xyz, box, periodic, edges)
        assert np.array_equal(ev, ev_ref) and np.array_equal(od, od_ref)
    hubs = np.arange(len(xyz))
    ev, od = oracle.count_4pcf_parity_hubs(xyz, box, periodic, edges, hubs)
    assert np.array_equal(ev, ev_ref) and np.array_equal(od, od_ref)


@pytest.mark.parametrize("periodic", [0, 1])
def test_4pcf_geometric_invariances(periodic):
    box = 30000
    xyz = catalogues.neyman_scott(700, box / 1024, 14, 50.0, 1.5, 51)
    edges = catalogues.linear_edges_lu(5.0, 6)
    ev, od = oracle.count_4pcf_parity(xyz, box, periodic, edges)
    assert ev.sum() > 1000 and np.abs(od).sum() > 0
    perm = np.random.default_rng(1).permutation(len(xyz))
    e2, o2 = oracle.count_4pcf_parity(xyz[perm], box, periodic, edges)
    assert np.array_equal(e2, ev) and np.array_equal(o2, od)
    # mirror: even unchanged, odd negated (Fig.1: mirror images have opposite V)
    e3, o3 = oracle.count_4pcf_parity(_mirror(xyz, box, periodic), box, periodic, edges)
    assert np.array_equal(e3, ev) and np.array_equal(o3, -od)
    # a cyclic axis permutation is a proper rotation: nothing changes
    e4, o4 = oracle.count_4pcf_parity(np.ascontiguousarray(xyz[:, [1, 2, 0]]), box, periodic, edges)
    assert np.array_equal(e4, ev) and np.array_equal(o4, od)
    # swapping two axes is a reflection
    e5, o5 = oracle.count_4pcf_parity(np.ascontiguousarray(xyz[:, [1, 0, 2]]), box, periodic, edges)
    assert np.array_equal(e5, ev) and np.array_equal(o5, -od)
    if periodic:
        moved = ((xyz.astype(np.int64) + np.array([4321, 29999, 15000])) % box).astype(np.int32)
        e6, o6 = oracle.count_4pcf_parity(moved, box, periodic, edges)
        assert np.array_equal(e6, ev) and np.array_equal(o6, od)


def test_4pcf_hub_ranges_sum_to_full():
    box = 30000
    xyz = catalogues.neyman_scott(500, box / 1024, 10, 50.0, 1.5, 61)
    edges = catalogues.linear_edges_lu(5.0, 5)
    g = oracle.graph(xyz, box, 1, edges)
    ev, od = oracle.count_4pcf_parity(xyz, box, 1, edges, g)
    cuts = [0, 7, 250, 499, 500]
    es = [oracle.count_4pcf_parity(xyz, box, 1, edges, g, a, b) for a, b in zip(cuts, cuts[1:])]
    assert np.array_equal(sum(e for e, _ in es), ev)
    assert np.array_equal(sum(o for _, o in es), od)


def test_degenerate_inputs():
    edges = [0, 100, 200]
    for n in (0, 1, 2):
        xyz = np.zeros((n, 3), dtype=np.int32) + 5
        assert oracle.count_3pcf(xyz, 1000, 1, edges).sum() == 0
        ev, od = oracle.count_4pcf_parity(xyz, 1000, 1, edges)
        assert ev.sum() == 0 and od.sum() == 0
    # three coincident points: one triangle in bin (0,0,0); one bin: no 4pCF configs
    xyz = np.full((3, 3), 7, dtype=np.int32)
    h = oracle.count_3pcf(xyz, 1000, 0, [0, 50])
    assert h.tolist() == [1]
    assert oracle.nconfig4(1) == 0 and oracle.nconfig4(2) == 0


# ---------------------------------------------------------------- per-hub (sampled) forms

def _np_hub_triangles(xyz, box, periodic, edges, hubs):
    nb = len(edges) - 1
    B, _ = fx.np_bins(xyz, box, periodic, edges)
    index = {c: n for n, c in enumerate(fx.configs3(nb))}
    hist = np.zeros(len(index), dtype=np.uint64)
    for h in hubs:
        spokes = np.nonzero(B[h] >= 0)[0]
        for j, k in itertools.combinations(spokes, 2):
            if B[j, k] >= 0:
                hist[index[tuple(sorted((int(B[h, j]), int(B[h, k]), int(B[j, k]))))]] += 1
    return hist


@pytest.mark.parametrize("periodic", [0, 1])
def test_3pcf_hubs_against_numpy_and_trace(periodic):
    box = 16000
    xyz = catalogues.neyman_scott(120, box / 1024, 6, 20.0, 1.5, 71 + periodic)
    edges = [0, 700, 1500, 2600, 4000]
    hubs = [0, 5, 5, 17, 119, 64]
    assert np.array_equal(oracle.count_3pcf_hubs(xyz, box, periodic, edges, hubs),
                          _np_hub_triangles(xyz, box, periodic, edges, hubs))
    # over all hubs every triangle is seen from each of its three vertices
    allh = oracle.count_3pcf_hubs(xyz, box, periodic, edges, np.arange(len(xyz)))
    assert np.array_equal(allh, 3 * oracle.count_3pcf(xyz, box, periodic, edges))


def test_3pcf_hubs_fixture():
    f = next(x for x in fx.triangle_fixtures() if x["name"] == "A")
    nb = len(f["edges"]) - 1
    h = oracle.count_3pcf_hubs(f["points"], f["box"], f["periodic"], f["edges"], np.arange(len(f["points"])))
    cfg = fx.configs3(nb)
    assert {cfg[k]: int(v) for k, v in enumerate(h) if v} == {c: 3 * n for c, n in f["expect"].items()}


def test_rows_and_parity_hubs_match_graph():
    box = 30000
    xyz = catalogues.neyman_scott(400, box / 1024, 8, 50.0, 1.5, 91)
    edges = catalogues.linear_edges_lu(5.0, 6)
    g = oracle.graph(xyz, box, 1, edges)
    for i in (0, 3, 399, 200):
        nbr, b = oracle.row(xyz, box, 1, edges, i)
        assert np.array_equal(nbr, g.nbr[g.row_ptr[i]:g.row_ptr[i + 1]])
        assert np.array_equal(b, g.bin[g.row_ptr[i]:g.row_ptr[i + 1]])
    e1, o1 = oracle.count_4pcf_parity_hubs(xyz, box, 1, edges, [7, 8, 9])
    e2, o2 = oracle.count_4pcf_parity(xyz, box, 1, edges, g, 7, 10)
    assert np.array_equal(e1, e2) and np.array_equal(o1, o2)


# ---------------------------------------------------------------- internal 2pCF

@pytest.mark.parametrize("periodic", [0, 1])
def test_2pcf_matches_numpy_pairs(periodic):
    box = 20000
    xyz = catalogues.neyman_scott(300, box / 1024, 10, 20.0, 1.5, 5 + periodic)
    edges = [0, 700, 1500, 2600, 4000, 6000]
    B, _ = fx.np_bins(xyz, box, periodic, edges)
    iu = np.triu_indices(len(xyz), 1)
    b = B[iu]
    ref = np.bincount(b[b >= 0], minlength=len(edges) - 1).astype(np.uint64)
    assert np.array_equal(oracle.count_2pcf(xyz, box, periodic, edges), ref)
    assert ref.sum() > 100


# ---------------------------------------------------------------- weighted counts (exact)

def test_weighted_counts_reduce_to_unweighted_and_scale():
    box = 20000
    xyz = catalogues.neyman_scott(200, box / 1024, 6, 30.0, 1.5, 8)
    edges = [0, 900, 1800, 3000]
    ones = np.ones(len(xyz), dtype=np.int16)
    assert oracle.count_2pcf_weighted(xyz, box, 1, edges, ones) == [int(v) for v in oracle.count_2pcf(xyz, box, 1, edges)]
    assert oracle.count_3pcf_weighted(xyz, box, 1, edges, ones) == [int(v) for v in oracle.count_3pcf(xyz, box, 1, edges)]
    big = np.full(len(xyz), 30000, dtype=np.int16)
    h = oracle.count_3pcf(xyz, box, 1, edges)
    assert oracle.count_3pcf_weighted(xyz, box, 1, edges, big) == [int(v) * 30000 ** 3 for v in h]


@pytest.mark.parametrize("periodic", [0, 1])
def test_weighted_counts_against_python_big_ints(periodic):
    box = 16000
    xyz = catalogues.neyman_scott(90, box / 1024, 5, 15.0, 1.5, 31 + periodic)
    edges = [0, 700, 1500, 2600, 4000]
    w = np.random.default_rng(4).integers(-32768, 32768, size=len(xyz)).astype(np.int16)
    B, _ = fx.np_bins(xyz, box, periodic, edges)
    nb = len(edges) - 1
    ref2 = [0] * nb
    for i, j in itertools.combinations(range(len(xyz)), 2):
        if B[i, j] >= 0:
            ref2[B[i, j]] += int(w[i]) * int(w[j])
    assert oracle.count_2pcf_weighted(xyz, box, periodic, edges, w) == ref2
    index = {c: n for n, c in enumerate(fx.configs3(nb))}
    ref3 = [0] * len(index)
    for i, j, k in itertools.combinations(range(len(xyz)), 3):
        b = (B[i, j], B[i, k], B[j, k])
        if min(b) >= 0:
            ref3[index[tuple(sorted(int(x) for x in b))]] += int(w[i]) * int(w[j]) * int(w[k])
    assert oracle.count_3pcf_weighted(xyz, box, periodic, edges, w) == ref3


def test_weighted_pair_sum_is_the_landy_szalay_numerator():
    # data weight +1, random weight -1 on the union: sum w_i w_j = DD - DR + RR,
    # with DR = (pairs of the union) - DD - RR from unweighted counts
    box = 30000
    d = catalogues.neyman_scott(300, box / 1024, 6, 50.0, 1.5, 2)
    r = catalogues.uniform(300, box / 1024, 3)
    edges = catalogues.linear_edges_lu(6.0, 5)
    u = np.vstack([d, r])
    w = np.concatenate([np.ones(300), -np.ones(300)]).astype(np.int16)
    dd = oracle.count_2pcf(d, box, 1, edges).astype(np.int64)
    rr = oracle.count_2pcf(r, box, 1, edges).astype(np.int64)
    tot = oracle.count_2pcf(u, box, 1, edges).astype(np.int64)
    dr = tot - dd - rr
    assert oracle.count_2pcf_weighted(u, box, 1, edges, w) == [int(v) for v in dd - dr + rr]
