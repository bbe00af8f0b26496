"""Internal 2pCF pair counts on the GPU against the oracle and, at full size,
against the closed form of a uniform periodic box (GRAMSCI v2 §III.3)."""
import math

import numpy as np
import pytest

import oracle
from cosmology_point_correlation_gb300 import as_uint64, catalogues, configs
from tests.gpu_util import gpu_graph

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("periodic", [0, 1])
@pytest.mark.parametrize("n", [1, 2, 17, 5003])
def test_2pcf_matches_oracle(periodic, n):
    box = catalogues.box_lattice(60.0)
    xyz = catalogues.neyman_scott(n, 60.0, max(1, n // 50), 50.0, 3.0, 9 + n)
    edges = catalogues.linear_edges_lu(10.0, 12)
    with gpu_graph(xyz, box, periodic, edges) as g:
        assert np.array_equal(as_uint64(g.count_2pcf()), oracle.count_2pcf(xyz, box, periodic, edges))


def test_2pcf_full_size_closed_form():
    w = configs.LARGE_3PCF
    with gpu_graph(w.points(), w.box_lu, True, w.edges_lu) as g:
        dd = as_uint64(g.count_2pcf()).astype(np.float64)
        assert dd.sum() * 2 == g.n_edges
    e = w.edges_lu.astype(np.float64)
    p = 4 * math.pi / 3 * (e[1:] ** 3 - e[:-1] ** 3) / float(w.box_lu) ** 3
    mean = math.comb(w.n, 2) * p
    z = (dd - mean) / np.sqrt(mean * (1 - p))
    assert np.all(np.abs(z) < 5), z
