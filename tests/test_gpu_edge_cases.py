"""Degenerate inputs through every count: empty and tiny catalogues, one bin,
isolated pairs and one triangle, device-resident and windowed (GRAMSCI v2
§II.1-§III.3, §III.5.3). Every result is checked against the oracle or a
value fixed by hand."""
import numpy as np
import pytest

import oracle
from cosmology_point_correlation_gb300 import as_int128, as_uint64, build_graph
from tests.gpu_util import torch_dev

pytestmark = pytest.mark.gpu

EDGES = [0, 1000, 2000, 3000, 4000]
BOX = 100_000


def _graph(xyz, window_edges=None, edges=EDGES, periodic=0):
    torch, dev = torch_dev()
    return build_graph(torch.from_numpy(np.asarray(xyz, dtype=np.int32).reshape(-1, 3)).to(dev), BOX, periodic,
                       edges, window_edges=window_edges)


def _all_counts(g, n, weights=None):
    torch, dev = torch_dev()
    out = {"pairs": as_uint64(g.count_2pcf()), "tri": as_uint64(g.count_3pcf())}
    e, o = g.count_4pcf_parity()
    out["par"] = (as_uint64(e), o.cpu().numpy())
    e, o = g.count_4pcf6()
    out["six"] = (as_uint64(e), o.cpu().numpy())
    w = np.ones(n, np.int16) if weights is None else weights
    g.set_weights(torch.from_numpy(w).to(dev))
    out["w2"] = as_int128(g.count_2pcf_weighted())
    out["w3"] = as_int128(g.count_3pcf_weighted())
    we, wo = g.count_4pcf6_weighted()
    out["w6"] = (as_int128(we), as_int128(wo))
    return out


@pytest.mark.parametrize("window_edges", [None, 1])
@pytest.mark.parametrize("n", [0, 1, 2])
def test_empty_and_tiny_catalogues(n, window_edges):
    # 0, 1 or 2 points far apart: no pair in range, every histogram zero
    xyz = np.array([[10, 10, 10], [90_000, 90_000, 90_000]], dtype=np.int32)[:n]
    with _graph(xyz, window_edges) as g:
        assert g.n == n and g.n_edges == 0
        c = _all_counts(g, n)
    assert not c["pairs"].any() and not c["tri"].any()
    assert not c["par"][0].any() and not c["par"][1].any()
    assert not c["six"][0].any() and not c["six"][1].any()
    assert not any(c["w2"]) and not any(c["w3"]) and not any(c["w6"][0]) and not any(c["w6"][1])


@pytest.mark.parametrize("window_edges", [None, 1])
def test_one_pair_and_one_triangle(window_edges):
    # a pair at distance 1500 (bin 1) and, far away, a (3,4,5)x500 triangle:
    # sides 1500, 2000, 2500 -> bins (1, 2, 2)
    xyz = [[10_000, 10_000, 10_000], [11_500, 10_000, 10_000],
           [50_000, 50_000, 50_000], [51_500, 50_000, 50_000], [50_000, 52_000, 50_000]]
    w = np.array([3, -2, 5, 7, -11], np.int16)
    with _graph(xyz, window_edges) as g:
        c = _all_counts(g, 5, w)
    assert c["pairs"].tolist() == [0, 2, 2, 0]                    # 1500, 1500 | 2000, 2500
    tri = np.zeros_like(c["tri"])
    tri[oracle.count_3pcf(np.asarray(xyz, np.int32), BOX, 0, EDGES).nonzero()] = 1
    assert np.array_equal(c["tri"], tri) and c["tri"].sum() == 1
    assert c["w2"] == oracle.count_2pcf_weighted(np.asarray(xyz, np.int32), BOX, 0, EDGES, w)
    assert c["w2"] == [0, 3 * -2 + 5 * 7, 5 * -11 + 7 * -11, 0]
    assert sum(c["w3"]) == 5 * 7 * -11
    assert not c["par"][0].any() and not c["six"][0].any()     # no four mutually adjacent points


def test_single_bin_and_coincident_points():
    # nbins = 1; coincident distinct points are a bin-0 edge (e_0 = 0). Four
    # coincident points and one 500 away: every pair is an edge, C(5,3) = 10
    # triangles and C(5,4) = 5 tetrahedra, each with at least three coincident
    # vertices, so of zero volume: even 5, odd 0
    xyz = np.array([[5000, 5000, 5000]] * 4 + [[5500, 5000, 5000]], dtype=np.int32)
    edges = [0, 1000]
    ref3 = oracle.count_3pcf(xyz, BOX, 0, edges)
    ref6e, ref6o = oracle.count_4pcf6(xyz, BOX, 0, edges)
    with _graph(xyz, edges=edges) as g:
        assert g.n_edges == 20
        assert as_uint64(g.count_2pcf()).tolist() == [10]
        assert np.array_equal(as_uint64(g.count_3pcf()), ref3) and ref3.sum() == 10
        e, o = g.count_4pcf6()
        assert np.array_equal(as_uint64(e), ref6e) and np.array_equal(o.cpu().numpy(), ref6o)
        assert ref6e.sum() == 5 and not ref6o.any()
        e, o = g.count_4pcf_parity()
        assert len(e) == 0 and len(o) == 0                      # C(1, 3) = 0 configurations
