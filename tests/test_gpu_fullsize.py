"""Full-size workloads, in the launch configuration the benchmark times.

The full histograms are beyond the oracle here (O(N^2) graph), so they are
checked on sampled outputs the oracle computes one by one, and by properties
that hold at any size:

* sampled rows N(i), by brute force over all N points (GRAMSCI v2 §II.1);
* sampled hubs: all triangles incident to the hub (§II.2 hub-and-spoke loop)
  and the hub's parity-4pCF contribution (§III.2), from brute-force rows;
* hub ranges covering [0, N) sum to the full histogram;
* triangles incident to all hubs = 3 x the histogram (every triangle has
  three vertices);
* the uniform periodic workload's total against the closed form
  C(N,3) p^2 15/32 (derivation in tests/test_oracle_stats.py); on a torus the
  first-order U-statistic variance vanishes and the relative scatter is
  sqrt(20 / (N^2 p)) (checked against a 48-seed ensemble at N = 2000);
* mirror symmetry: 3pCF and even unchanged, odd negated (Fig.1).
"""
import math

import numpy as np
import pytest

import oracle
from cosmology_point_correlation_gb300 import as_uint64, configs
from tests.gpu_util import gpu_graph, mirror

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

SAMPLE_HUBS = 24


def _sample(n, seed):
    return np.random.default_rng(seed).choice(n, size=SAMPLE_HUBS, replace=False)


def _check_rows(g, xyz, w, ids):
    rp, nbr, b = (t.cpu().numpy() for t in g.export_rows(ids))
    for t, i in enumerate(ids):
        rn, rb = oracle.row(xyz, w.box_lu, int(w.periodic), w.edges_lu, int(i))
        assert np.array_equal(nbr[rp[t]:rp[t + 1]], rn), f"row {i}"
        assert np.array_equal(b[rp[t]:rp[t + 1]], rb), f"bins of row {i}"


@pytest.mark.parametrize("name", ["clustered_3pcf_data", "clustered_3pcf_randoms", "large_3pcf", "bao_3pcf"])
def test_3pcf_workload_sampled(name):
    w = configs.ALL[name]
    xyz = w.points()
    with gpu_graph(xyz, w.box_lu, w.periodic, w.edges_lu) as g:
        full = as_uint64(g.count_3pcf())
        assert full.sum() > 0
        hubs = _sample(len(xyz), w.seed)
        _check_rows(g, xyz, w, hubs[:8])
        ref = oracle.count_3pcf_hubs(xyz, w.box_lu, int(w.periodic), w.edges_lu, hubs)
        assert np.array_equal(as_uint64(g.count_3pcf_hubs(hubs)), ref)
        # properties at full size
        cut = len(xyz) // 3
        parts = as_uint64(g.count_3pcf(0, cut)) + as_uint64(g.count_3pcf(cut, len(xyz)))
        assert np.array_equal(parts, full)
        if name != "bao_3pcf":
            allh = as_uint64(g.count_3pcf_hubs(np.arange(len(xyz), dtype=np.int32)))
            assert np.array_equal(allh, 3 * full)


def test_large_uniform_total_closed_form_and_mirror():
    w = configs.LARGE_3PCF
    xyz = w.points()
    with gpu_graph(xyz, w.box_lu, True, w.edges_lu) as g:
        full = as_uint64(g.count_3pcf())
    n = len(xyz)
    p = 4 * math.pi / 3 * (w.edges_lu[-1] / w.box_lu) ** 3
    expect = math.comb(n, 3) * p * p * 15 / 32
    sigma = expect * math.sqrt(20 / (n * n * p))
    assert abs(int(full.sum()) - expect) < 5 * sigma
    with gpu_graph(mirror(xyz, w.box_lu, True), w.box_lu, True, w.edges_lu) as g:
        assert np.array_equal(as_uint64(g.count_3pcf()), full)


def test_parity_workload_sampled_and_mirror():
    w = configs.PARITY_4PCF
    xyz = w.points()
    with gpu_graph(xyz, w.box_lu, True, w.edges_lu) as g:
        ev, od = g.count_4pcf_parity()
        ev, od = as_uint64(ev), od.cpu().numpy()
        assert ev.sum() > 0
        hubs = _sample(len(xyz), w.seed)
        _check_rows(g, xyz, w, hubs[:8])
        re, ro = oracle.count_4pcf_parity_hubs(xyz, w.box_lu, 1, w.edges_lu, hubs)
        e, o = g.count_4pcf_parity_hubs(hubs)
        assert np.array_equal(as_uint64(e), re) and np.array_equal(o.cpu().numpy(), ro)
        cut = len(xyz) // 2
        e1, o1 = g.count_4pcf_parity(0, cut)
        e2, o2 = g.count_4pcf_parity(cut, len(xyz))
        assert np.array_equal(as_uint64(e1) + as_uint64(e2), ev)
        assert np.array_equal(o1.cpu().numpy() + o2.cpu().numpy(), od)
    with gpu_graph(mirror(xyz, w.box_lu, True), w.box_lu, True, w.edges_lu) as g:
        me, mo = g.count_4pcf_parity()
        assert np.array_equal(as_uint64(me), ev) and np.array_equal(mo.cpu().numpy(), -od)
