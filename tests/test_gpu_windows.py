"""Out-of-core row windows (GRAMSCI v2 §III.5.3): the edge arrays in pinned
host memory, queries run as tiles of (hub window, spoke window) for the 3pCF
and of (hub window, spoke windows c1 <= c2) for the 4pCF. Every triangle and
clique lands in exactly one tile, so the windowed results equal the
device-resident ones and the oracle bit for bit, for any window size."""
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


@pytest.mark.parametrize("walk", ["map", "mapgroup", "warp"])
@pytest.mark.parametrize("periodic", [0, 1])
@pytest.mark.parametrize("frac", [1.0, 0.3, 0.05, 0.0])
def test_windowed_graph_and_3pcf_match_oracle(periodic, frac, walk, monkeypatch):
    # frac of the edges per window; 0 -> one cell per window. Window tiles run
    # the byte-map walks (one or four spokes per warp) or the bitmap walk.
    monkeypatch.setenv("GS_COUNT3_WALK", walk)
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


@pytest.mark.parametrize("periodic", [0, 1])
@pytest.mark.parametrize("frac", [0.2, 0.0])
def test_windowed_four_point_counts_match_oracle(periodic, frac):
    # tiles over (hub window, spoke windows c1 <= c2): parity, six-bin and
    # weighted six-bin counts equal the oracle for several window sizes
    torch, dev = torch_dev()
    n = 8_000
    L = 500.0 * (n / 200_000) ** (1 / 3)
    box = catalogues.box_lattice(L)
    xyz = catalogues.neyman_scott(n, L, n // 50, 50.0, 3.0, 40 + periodic)
    e8 = catalogues.linear_edges_lu(20.0, 8)
    e4 = catalogues.linear_edges_lu(20.0, 4)
    ref_e, ref_o = oracle.count_4pcf_parity(xyz, box, periodic, e8)
    assert ref_e.sum() > 1000
    g8 = oracle.graph(xyz, box, periodic, e8)
    with _graph(xyz, box, periodic, e8, max(1, int(frac * g8.n_edges))) as g:
        assert g.windows()[0] > 2
        ev, od = g.count_4pcf_parity()
        assert np.array_equal(as_uint64(ev), ref_e) and np.array_equal(od.cpu().numpy(), ref_o)
        cut = n // 2
        e1, o1 = g.count_4pcf_parity(0, cut)
        e2, o2 = g.count_4pcf_parity(cut, n)
        assert np.array_equal(as_uint64(e1) + as_uint64(e2), ref_e)
        assert np.array_equal(o1.cpu().numpy() + o2.cpu().numpy(), ref_o)
    s_e, s_o = oracle.count_4pcf6(xyz, box, periodic, e4)
    w = np.random.default_rng(6).integers(-32767, 32768, size=n).astype(np.int16)
    ref_w = oracle.count_4pcf6_weighted(xyz, box, periodic, e4, w)
    g4 = oracle.graph(xyz, box, periodic, e4)
    with _graph(xyz, box, periodic, e4, max(1, int(frac * g4.n_edges))) as g:
        assert g.windows()[0] > 2
        ev, od = g.count_4pcf6()
        assert np.array_equal(as_uint64(ev), s_e) and np.array_equal(od.cpu().numpy(), s_o)
        g.set_weights(torch.from_numpy(w).to(dev))
        we, wo = g.count_4pcf6_weighted()
        assert (as_int128(we), as_int128(wo)) == ref_w


def test_windowed_limits_and_environment_override():
    torch, dev = torch_dev()
    w = configs.TINY_3PCF
    xyz = w.points()
    with _graph(xyz, w.box_lu, 1, w.edges_lu, 10_000) as g:
        with pytest.raises(GramsciError, match="windowed"):
            g.count_3pcf_hubs([0, 1])
        with pytest.raises(GramsciError, match="windowed"):
            g.count_4pcf_parity_hubs([0, 1])
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


def test_windowed_large_hubs_equal_resident():
    # a hub with 700 neighbours on a shell: the global-workspace kernels of
    # both 4pCF counts run per tile; windowed equals device-resident
    rng = np.random.default_rng(8)
    R = 20000
    v = rng.normal(size=(700, 3))
    v *= (0.9 * R * (0.5 + 0.5 * rng.uniform(size=(700, 1)))) / np.linalg.norm(v, axis=1, keepdims=True)
    xyz = (np.vstack([[[0, 0, 0]], np.rint(v)]) + 25000).astype(np.int32)
    edges = [0, 8000, 12000, 16000, R]
    with _graph(xyz, 50000, 0, edges) as g:
        assert g.max_degree > 512
        pe, po = (t.cpu().numpy() for t in g.count_4pcf_parity())
        se, so = (t.cpu().numpy() for t in g.count_4pcf6())
    with _graph(xyz, 50000, 0, edges, 1) as g:
        assert g.windows()[0] > 2
        e, o = (t.cpu().numpy() for t in g.count_4pcf_parity())
        assert np.array_equal(e, pe) and np.array_equal(o, po)
        e, o = (t.cpu().numpy() for t in g.count_4pcf6())
        assert np.array_equal(e, se) and np.array_equal(o, so)


@pytest.mark.slow
def test_build_switches_to_windows_when_the_graph_does_not_fit():
    # §III.5.3: chunked mode is selected at run time when the graph exceeds the
    # free device memory. Hold all but 3 GB of it, then build the 2M-point
    # uniform graph (5.4 GB of CSR): it must come out windowed and count the same.
    torch, dev = torch_dev()
    w = configs.LARGE_3PCF
    xyz = w.points()
    with _graph(xyz, w.box_lu, True, w.edges_lu) as g:
        assert g.windows()[0] == 0
        full = as_uint64(g.count_3pcf())
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    free, _ = torch.cuda.mem_get_info()
    hold = torch.empty(max(free - (3 << 30), 0), dtype=torch.uint8, device=dev)
    try:
        with _graph(xyz, w.box_lu, True, w.edges_lu) as g:
            nw, wmax = g.windows()
            assert nw > 2 and wmax < g.n_edges
            assert np.array_equal(as_uint64(g.count_3pcf()), full)
    finally:
        del hold
        torch.cuda.empty_cache()
