"""Neighbour graph on the GPU equals the brute-force oracle graph exactly
(GRAMSCI v2 §II.1, Eq.(1): sorted rows with a bin byte per neighbour)."""
import numpy as np
import pytest

from cosmology_point_correlation_gb300 import catalogues, configs
from tests import fixtures as fx
from tests.gpu_util import assert_graph_equal, gpu_csr

pytestmark = pytest.mark.gpu


def test_tiny_config():
    w = configs.TINY_3PCF
    ref = assert_graph_equal(w.points(), w.box_lu, w.periodic, w.edges_lu)
    assert ref.n_edges > 100_000


@pytest.mark.parametrize("periodic", [0, 1])
def test_clustered(periodic):
    box = catalogues.box_lattice(150.0)
    xyz = catalogues.neyman_scott(20_000, 150.0, 400, 50.0, 3.0, 77 + periodic)
    assert_graph_equal(xyz, box, periodic, catalogues.linear_edges_lu(9.0, 12))


@pytest.mark.parametrize("case", list(fx.pair_bin_cases()))
def test_pair_rule_fixtures(case):
    box, periodic, edges, p, q, expect = case
    rp, nbr, b, _ = gpu_csr(np.array([p, q], dtype=np.int32), box, periodic, edges)
    if expect < 0:
        assert rp.tolist() == [0, 0, 0]
    else:
        assert rp.tolist() == [0, 1, 2] and nbr.tolist() == [1, 0] and b.tolist() == [expect, expect]


def test_inner_edge_above_zero():
    box = catalogues.box_lattice(40.0)
    xyz = catalogues.uniform(3000, 40.0, 5)
    assert_graph_equal(xyz, box, 1, [3000, 5000, 6500, 9000])


@pytest.mark.parametrize("periodic,rmax", [(1, 9000), (1, 10000), (0, 25000), (0, 15000)])
def test_few_cells_per_axis(periodic, rmax):
    # box 20000: 2 cells per axis (periodic duplicates are de-duplicated) or 1
    xyz = catalogues.uniform(1500, 20000 / 1024, 9)
    assert_graph_equal(xyz, 20000, periodic, [0, rmax // 3, rmax])


def test_dense_cells_span_several_tiles():
    # ~1250 points per cell: more than one staged home batch and candidate tile
    xyz = catalogues.uniform(10_000, 20000 / 1024, 13)
    assert_graph_equal(xyz, 20000, 1, [0, 3000, 6000, 9000])


@pytest.mark.parametrize("n", [0, 1, 2, 3, 33])
def test_tiny_and_degenerate_inputs(n):
    xyz = np.full((n, 3), 1234, dtype=np.int32)       # coincident points: bin 0 edges
    assert_graph_equal(xyz, 50000, 1, [0, 100, 200])
    xyz = catalogues.uniform(n, 50000 / 1024, 3)
    assert_graph_equal(xyz, 50000, 0, [0, 100, 20000])


def test_rows_sorted_and_symmetric_on_clustered_open_box():
    w = configs.CLUSTERED_3PCF_D
    xyz = w.points(n=30_000)
    rp, nbr, b, _ = gpu_csr(xyz, w.box_lu, 0, w.edges_lu)
    n = len(xyz)
    rows = np.repeat(np.arange(n), np.diff(rp))
    assert np.all(nbr != rows)
    same_row = rows[1:] == rows[:-1]
    assert np.all(np.diff(nbr)[same_row] > 0)
    key = rows.astype(np.int64) * n + nbr
    rkey = nbr.astype(np.int64) * n + rows
    order = np.argsort(key)
    pos = np.searchsorted(key[order], rkey)
    assert np.array_equal(key[order][pos], rkey)
    assert np.array_equal(b[order][pos], b)


@pytest.mark.parametrize("periodic", [0, 1])
def test_hub_work_matches_the_oracle_graph(periodic):
    # f_i = |{j in N(i): j > i}| and w_i = sum of f_j over those j, in the
    # graph's internal order (the input put in that order first)
    import oracle
    from tests.gpu_util import gpu_graph
    box = catalogues.box_lattice(100.0)
    xyz = catalogues.neyman_scott(8000, 100.0, 160, 50.0, 3.0, 31 + periodic)
    edges = catalogues.linear_edges_lu(10.0, 6)
    with gpu_graph(xyz, box, periodic, edges) as g:
        perm = g.export_perm().cpu().numpy()
    xg = np.ascontiguousarray(xyz[perm])
    ref = oracle.graph(xg, box, periodic, edges)
    n = len(xg)
    f = np.array([(ref.nbr[ref.row_ptr[i]:ref.row_ptr[i + 1]] > i).sum() for i in range(n)])
    w = np.array([f[ref.nbr[ref.row_ptr[i]:ref.row_ptr[i + 1]][ref.nbr[ref.row_ptr[i]:ref.row_ptr[i + 1]] > i]].sum()
                  for i in range(n)])
    with gpu_graph(xg, box, periodic, edges) as g:
        gf, gw = (t.cpu().numpy() for t in g.hub_work())
        st = g.stats()
    assert np.array_equal(gf, f) and np.array_equal(gw, w)
    assert gw.sum() == st["spoke_walk"] and gf.max() == st["max_forward"]
