"""Per-hub entry points and row export on the GPU against the oracle (small
catalogues): the kernels of the full counts, restricted to listed hubs."""
import numpy as np
import pytest

import oracle
from cosmology_point_correlation_gb300 import as_uint64, catalogues
from tests.gpu_util import gpu_graph

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("periodic", [0, 1])
def test_3pcf_hubs_and_trace(periodic):
    box = catalogues.box_lattice(100.0)
    xyz = catalogues.neyman_scott(8000, 100.0, 160, 50.0, 3.0, 44 + periodic)
    edges = catalogues.linear_edges_lu(10.0, 12)
    hubs = np.random.default_rng(1).integers(0, len(xyz), size=300)
    ref = oracle.count_3pcf_hubs(xyz, box, periodic, edges, hubs)
    with gpu_graph(xyz, box, periodic, edges) as g:
        assert np.array_equal(as_uint64(g.count_3pcf_hubs(hubs)), ref)
        allh = as_uint64(g.count_3pcf_hubs(np.arange(len(xyz))))
        assert np.array_equal(allh, 3 * as_uint64(g.count_3pcf()))
        assert as_uint64(g.count_3pcf_hubs([])).sum() == 0


def test_3pcf_hubs_on_rows_longer_than_the_table():
    rng = np.random.default_rng(3)
    R = 40000
    v = rng.normal(size=(2300, 3))
    v *= (0.45 * R * rng.uniform(0, 1, size=(2300, 1)) ** (1 / 3)) / np.linalg.norm(v, axis=1, keepdims=True)
    xyz = (v + 100000).astype(np.int32)
    edges = [0, 9000, 21000, 33000, R]
    hubs = [0, 1, 1000, 2299]
    ref = oracle.count_3pcf_hubs(xyz, 300000, 0, edges, hubs)
    with gpu_graph(xyz, 300000, 0, edges) as g:
        assert np.array_equal(as_uint64(g.count_3pcf_hubs(hubs)), ref)


@pytest.mark.parametrize("periodic", [0, 1])
def test_parity_hubs(periodic):
    box = catalogues.box_lattice(60.0)
    xyz = catalogues.neyman_scott(5000, 60.0, 100, 50.0, 3.0, 12 + periodic)
    edges = catalogues.linear_edges_lu(10.0, 8)
    hubs = np.random.default_rng(2).integers(0, len(xyz), size=200)
    ref_e, ref_o = oracle.count_4pcf_parity_hubs(xyz, box, periodic, edges, hubs)
    with gpu_graph(xyz, box, periodic, edges) as g:
        e, o = g.count_4pcf_parity_hubs(hubs)
        assert np.array_equal(as_uint64(e), ref_e) and np.array_equal(o.cpu().numpy(), ref_o)


def test_export_rows():
    box = catalogues.box_lattice(80.0)
    xyz = catalogues.neyman_scott(6000, 80.0, 120, 50.0, 3.0, 3)
    edges = catalogues.linear_edges_lu(9.0, 9)
    ids = [0, 5999, 17, 17, 3000]
    with gpu_graph(xyz, box, 1, edges) as g:
        rp, nbr, b = (t.cpu().numpy() for t in g.export_rows(ids))
    for t, i in enumerate(ids):
        rn, rb = oracle.row(xyz, box, 1, edges, i)
        assert np.array_equal(nbr[rp[t]:rp[t + 1]], rn) and np.array_equal(b[rp[t]:rp[t + 1]], rb)


def test_hub_index_out_of_range_is_rejected():
    from cosmology_point_correlation_gb300 import GramsciError
    xyz = catalogues.uniform(500, 20.0, 1)
    with gpu_graph(xyz, catalogues.box_lattice(20.0), 1, [0, 1000, 2000]) as g:
        for bad in ([500], [-1], [3, 700]):
            with pytest.raises(GramsciError, match="outside"):
                g.count_3pcf_hubs(bad)
            with pytest.raises(GramsciError, match="outside"):
                g.export_rows(bad)
