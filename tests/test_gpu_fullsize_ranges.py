"""Full-size workloads: the counts the benchmark times, on contiguous hub
ranges, against the oracle over the same hubs.

The GRAMSCI v2 paper checks its GPU counts against the CPU code on the
production-size run and finds every binned count equal (§IV.8). Here the full
histograms are beyond the oracle (its graph is O(N^2)), so each workload is
checked on hub ranges:

* the input is put in the graph's own (cell) order with the exported
  permutation, so hub i of the library is point i for the oracle;
* the oracle gets brute-force rows (over all N points) for the hubs of the
  range only; its hub loops need no other row, because they test the closing
  sides from coordinates (§II.2 for triangles, §III.2 for the spoke triples);
* the library counts the same range with the call and walk the benchmark
  uses (`count_3pcf(b, e)`, `count_4pcf_parity(b, e)`, `count_4pcf6(b, e)`),
  and the histograms must be equal bit for bit;
* the ranges are chosen from the per-hub work the library exports: one
  around the hub with the longest merge-walk (the densest cluster, where
  rows are longest), one around the hub of largest forward degree, one in
  the middle of the catalogue;
* the three ranges plus the rest of [0, N) add up to the full-catalogue
  launch, which ties the range launches to the one the benchmark times.
"""
import dataclasses

import numpy as np
import pytest

import oracle
from cosmology_point_correlation_gb300 import as_uint64, configs
from tests.gpu_util import gpu_graph

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _part_graph(xyz, w, periodic, ranges):
    """Oracle graph holding brute-force rows for the hubs of `ranges` only."""
    n = len(xyz)
    deg = np.zeros(n, dtype=np.int64)
    nbrs, bins = [], []
    for b, e in sorted(ranges):
        for i in range(b, e):
            r, rb = oracle.row(xyz, w.box_lu, periodic, w.edges_lu, i)
            deg[i] = len(r)
            nbrs.append(r)
            bins.append(rb)
    row_ptr = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(deg, out=row_ptr[1:])
    nbr = np.concatenate(nbrs).astype(np.int32) if nbrs else np.zeros(0, np.int32)
    bn = np.concatenate(bins).astype(np.uint8) if bins else np.zeros(0, np.uint8)
    return oracle.Graph(row_ptr, nbr, bn)


def _around(i, half, n):
    b = max(0, min(int(i) - half, n - 2 * half))
    return b, min(n, b + 2 * half)


def _disjoint(ranges):
    out = []
    for b, e in sorted(set(ranges)):
        if out and b < out[-1][1]:
            b = out[-1][1]
        if b < e:
            out.append((b, e))
    return out


def _ranges(g, half):
    f, wk = (t.cpu().numpy() for t in g.hub_work())
    n = len(f)
    return _disjoint([_around(np.argmax(wk), half, n), _around(np.argmax(f), half, n),
                      _around(n // 2, half, n)]), f, wk


def _complement(ranges, n):
    cuts = [0] + [x for r in ranges for x in r] + [n]
    return [(cuts[k], cuts[k + 1]) for k in range(0, len(cuts), 2) if cuts[k] < cuts[k + 1]]


# hubs per range (half-width): the oracle's cost grows with f^2 per hub
HALF = {"clustered_3pcf_data": 100, "clustered_3pcf_randoms": 100, "large_3pcf": 48, "bao_3pcf": 24}


@pytest.mark.parametrize("name", list(HALF))
def test_3pcf_hub_ranges_of_the_full_workload(name):
    w = configs.ALL[name]
    xyz = w.points()
    p = int(w.periodic)
    with gpu_graph(xyz, w.box_lu, p, w.edges_lu) as g:
        perm = g.export_perm().cpu().numpy()
        ranges, f, wk = _ranges(g, HALF[name])
        full = as_uint64(g.count_3pcf())
        got = {r: as_uint64(g.count_3pcf(*r)) for r in ranges}
        rest = [as_uint64(g.count_3pcf(*r)) for r in _complement(ranges, len(xyz))]
    assert np.array_equal(sum(got.values()) + sum(rest), full)
    xg = np.ascontiguousarray(xyz[perm])
    part = _part_graph(xg, w, p, ranges)
    for (b, e), h in got.items():
        ref = oracle.count_3pcf(xg, w.box_lu, p, w.edges_lu, g=part, hub_begin=b, hub_end=e)
        assert ref.sum() > 0, (b, e)
        assert np.array_equal(h, ref), f"{name}: hubs [{b}, {e}) differ from the oracle"
    # the densest range really holds the longest rows of the catalogue
    assert any(b <= np.argmax(wk) < e for b, e in ranges)
    assert any(b <= np.argmax(f) < e for b, e in ranges)


@pytest.mark.parametrize("walk", ["warp", "group", "map", "mapgroup"])
@pytest.mark.parametrize("name", ["clustered_3pcf_data", "large_3pcf", "bao_3pcf"])
def test_3pcf_hub_ranges_every_walk(name, walk, monkeypatch):
    # the benchmark's walk is chosen from the graph; every walk must give the
    # oracle's histogram on the full-size graph
    monkeypatch.setenv("GS_COUNT3_WALK", walk)
    w = configs.ALL[name]
    xyz = w.points()
    p = int(w.periodic)
    with gpu_graph(xyz, w.box_lu, p, w.edges_lu) as g:
        perm = g.export_perm().cpu().numpy()
        ranges, _, _ = _ranges(g, HALF[name] // 2)
        got = {r: as_uint64(g.count_3pcf(*r)) for r in ranges}
    xg = np.ascontiguousarray(xyz[perm])
    part = _part_graph(xg, w, p, ranges)
    for (b, e), h in got.items():
        assert np.array_equal(h, oracle.count_3pcf(xg, w.box_lu, p, w.edges_lu, g=part, hub_begin=b, hub_end=e))


def _parity_ranges(g, half):
    f, _ = (t.cpu().numpy() for t in g.hub_work())
    rp, _, _ = g.export_rows(g.export_perm())
    deg = np.diff(rp.cpu().numpy())
    n = len(deg)
    return _disjoint([_around(np.argmax(deg), half, n), _around(np.argmax(f), half, n),
                      _around(n // 2, half, n)]), deg


def test_parity_hub_ranges_of_the_full_workload():
    w = configs.PARITY_4PCF
    xyz = w.points()
    with gpu_graph(xyz, w.box_lu, 1, w.edges_lu) as g:
        perm = g.export_perm().cpu().numpy()
        ranges, deg = _parity_ranges(g, 100)
        ev, od = g.count_4pcf_parity()
        full_e, full_o = as_uint64(ev), od.cpu().numpy()
        got = {}
        for r in ranges:
            e, o = g.count_4pcf_parity(*r)
            got[r] = (as_uint64(e), o.cpu().numpy())
        rest_e, rest_o = 0, 0
        for r in _complement(ranges, len(xyz)):
            e, o = g.count_4pcf_parity(*r)
            rest_e, rest_o = rest_e + as_uint64(e), rest_o + o.cpu().numpy()
    assert np.array_equal(sum(v[0] for v in got.values()) + rest_e, full_e)
    assert np.array_equal(sum(v[1] for v in got.values()) + rest_o, full_o)
    xg = np.ascontiguousarray(xyz[perm])
    part = _part_graph(xg, w, 1, ranges)
    for (b, e), (he, ho) in got.items():
        re, ro = oracle.count_4pcf_parity(xg, w.box_lu, 1, w.edges_lu, g=part, hub_begin=b, hub_end=e)
        assert re.sum() > 0
        assert np.array_equal(he, re) and np.array_equal(ho, ro), f"parity: hubs [{b}, {e}) differ"
    assert any(b <= np.argmax(deg) < e for b, e in ranges)


def test_six_bin_hub_ranges_of_the_parity_workload():
    # the six-bin 4pCF the benchmark times on the parity catalogue with 4 bins
    w = dataclasses.replace(configs.PARITY_4PCF, nbins=4)
    xyz = w.points()
    with gpu_graph(xyz, w.box_lu, 1, w.edges_lu) as g:
        perm = g.export_perm().cpu().numpy()
        ranges, _, _ = _ranges(g, 60)
        ev, od = g.count_4pcf6()
        full_e, full_o = as_uint64(ev), od.cpu().numpy()
        got = {}
        for r in ranges:
            e, o = g.count_4pcf6(*r)
            got[r] = (as_uint64(e), o.cpu().numpy())
        rest_e, rest_o = 0, 0
        for r in _complement(ranges, len(xyz)):
            e, o = g.count_4pcf6(*r)
            rest_e, rest_o = rest_e + as_uint64(e), rest_o + o.cpu().numpy()
    assert np.array_equal(sum(v[0] for v in got.values()) + rest_e, full_e)
    assert np.array_equal(sum(v[1] for v in got.values()) + rest_o, full_o)
    xg = np.ascontiguousarray(xyz[perm])
    part = _part_graph(xg, w, 1, ranges)
    for (b, e), (he, ho) in got.items():
        re, ro = oracle.count_4pcf6(xg, w.box_lu, 1, w.edges_lu, g=part, hub_begin=b, hub_end=e)
        assert re.sum() > 0
        assert np.array_equal(he, re) and np.array_equal(ho, ro), f"six-bin: hubs [{b}, {e}) differ"
