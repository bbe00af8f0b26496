"""Out-of-core row windows (GRAMSCI v2 §III.5.3): the edge arrays in pinned
host memory, queries run as (hub window, spoke window) tiles. Every triangle
lands in exactly one tile, so the windowed results equal the device-resident
ones and the oracle bit for bit, for any window size."""
import os

import numpy as np
import pytest

import oracle
from cosmology_point_correlation_gb300 import GramsciError, as_int128, as_uint64, build_graph, catalogues, configs
from tests.gpu_util import torch_dev

pytestmark = pytest.mark.gpu


def _graph(xyz, box, periodic, edges, window_edges=None):
    torch, dev = torch_dev()
    return build_graph(torch.from_numpy(np.ascontiguousarray(xyz, dtype=np.int32)).to(dev), box, periodic, edges,
                       window_edges=window_edges)


def _clustered(n, seed, periodic):
    box = catalogues.box_lattice(120.0)
    xyz = catalogues.neyman_scott(n, 120.0, n // 50, 50.0, 3.0, seed + periodic)
    return xyz, box, catalogues.linear_edges_lu(10.0, 15)


@pytest.mark.parametrize("periodic", [0, 1])
@pytest.mark.parametrize("frac", [1.0, 0.3, 0.05, 0.0])
def test_windowed_graph_and_3pcf_match_oracle(periodic, frac):
    # frac of the edges per window; 0 -> one cell per window
    xyz, box, edges = _clustered(20_011, 5, periodic)
    ref = oracle.graph(xyz, box, periodic, edges)
    hist_ref = oracle.count_3pcf(xyz, box, periodic, edges, ref)
    with _graph(xyz, box, periodic, edges, max(1, int(frac * ref.n_edges))) as g:
        nw, wmax = g.windows()
        assert nw >= (1 if frac == 1.0 else 2)
        assert wmax <= max(1, int(frac * ref.n_edges)) or frac == 0.0
        rp, nbr, b = (t.cpu().numpy() for t in g.export_csr())
        assert np.array_equal(rp, ref.row_ptr) and np.array_equal(nbr, ref.nbr) and np.array_equal(b, ref.bin)
        assert np.array_equal(as_uint64(g.count_3pcf()), hist_ref)
        assert np.array_equal(as_uint64(g.count_2pcf()), oracle.count_2pcf(xyz, box, periodic, edges, ref))
        # hub ranges that cut across windows still add up
        n = len(xyz)
        parts = [as_uint64(g.count_3pcf(a, c)) for a, c in [(0, n // 3), (n // 3, n // 3 + 17), (n // 3 + 17, n)]]
        assert np.array_equal(np.sum(parts, axis=0, dtype=np.uint64), hist_ref)


def test_windowed_weighted_counts():
    torch, dev = torch_dev()
    xyz, box, edges = _clustered(12_000, 9, 1)
    w = np.random.default_rng(4).integers(-32767, 32768, size=len(xyz)).astype(np.int16)
    with _graph(xyz, box, 1, edges, 50_000) as g:
        assert g.windows()[0] > 3
        g.set_weights(torch.from_numpy(w).to(dev))
        assert as_int128(g.count_3pcf_weighted()) == oracle.count_3pcf_weighted(xyz, box, 1, edges, w)
        assert as_int128(g.count_2pcf_weighted()) == oracle.count_2pcf_weighted(xyz, box, 1, edges, w)


def test_windowed_limits_and_environment_override():
    torch, dev = torch_dev()
    w = configs.TINY_3PCF
    xyz = w.points()
    with _graph(xyz, w.box_lu, 1, w.edges_lu, 10_000) as g:
        with pytest.raises(GramsciError, match="windowed"):
            g.count_4pcf_parity()
        with pytest.raises(GramsciError, match="windowed"):
            g.count_4pcf6()
        with pytest.raises(GramsciError, match="windowed"):
            g.count_3pcf_hubs([0, 1])
        ref = as_uint64(g.count_3pcf())
    with pytest.raises(GramsciError):
        _graph(xyz, w.box_lu, 1, w.edges_lu, 0)
    os.environ["GS_WINDOW_EDGES"] = "20000"
    try:
        with _graph(xyz, w.box_lu, 1, w.edges_lu) as g:
            assert g.windows()[0] > 1
            assert np.array_equal(as_uint64(g.count_3pcf()), ref)
    finally:
        del os.environ["GS_WINDOW_EDGES"]
    with _graph(xyz, w.box_lu, 1, w.edges_lu) as g:
        assert g.windows()[0] == 0
        assert np.array_equal(as_uint64(g.count_3pcf()), ref)
    # empty catalogue
    with _graph(np.zeros((0, 3), np.int32), w.box_lu, 1, w.edges_lu, 100) as g:
        assert not as_uint64(g.count_3pcf()).any()


@pytest.mark.slow
@pytest.mark.parametrize("windows", [2, 8])
def test_large_workload_windowed_equals_resident(windows):
    w = configs.LARGE_3PCF
    xyz = w.points()
    with _graph(xyz, w.box_lu, True, w.edges_lu) as g:
        full = as_uint64(g.count_3pcf())
        pairs = as_uint64(g.count_2pcf())
        e = g.n_edges
    with _graph(xyz, w.box_lu, True, w.edges_lu, e // windows + 1) as g:
        assert g.windows()[0] >= windows
        assert np.array_equal(as_uint64(g.count_3pcf()), full)
        assert np.array_equal(as_uint64(g.count_2pcf()), pairs)
