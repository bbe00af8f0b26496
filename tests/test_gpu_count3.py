"""3pCF triangle histograms on the GPU equal the oracle bit for bit
(GRAMSCI v2 §II.2, §III.1; configurations as in §V.1 Fig.8)."""
import numpy as np
import pytest

import oracle
from cosmology_point_correlation_gb300 import as_uint64, catalogues, configs, count_3pcf_from_host
from tests import fixtures as fx
from tests.gpu_util import gpu_3pcf, gpu_graph, mirror

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, params=["warp", "group", "map", "mapgroup"])
def walk_mode(request, monkeypatch):
    """Every test of this module runs with each spoke walk of the 3pCF count:
    one or four spokes per warp over a bitmap of the hub's keys, and one or
    four spokes per warp over a byte map of the keys' bins (read at each
    launch)."""
    monkeypatch.setenv("GS_COUNT3_WALK", request.param)
    return request.param


def test_tiny_config():
    w = configs.TINY_3PCF
    xyz = w.points()
    ref = oracle.count_3pcf(xyz, w.box_lu, 1, w.edges_lu)
    assert ref.sum() > 600_000
    assert np.array_equal(gpu_3pcf(xyz, w.box_lu, 1, w.edges_lu), ref)


@pytest.mark.parametrize("fixture", list(fx.triangle_fixtures()), ids=lambda f: f["name"])
def test_fixtures(fixture):
    f = fixture
    nb = len(f["edges"]) - 1
    hist = gpu_3pcf(f["points"], f["box"], f["periodic"], f["edges"])
    cfg = fx.configs3(nb)
    assert {cfg[k]: int(v) for k, v in enumerate(hist) if v} == f["expect"]


@pytest.mark.parametrize("periodic", [0, 1])
@pytest.mark.parametrize("n", [5_000, 20_011])
def test_clustered(periodic, n):
    box = catalogues.box_lattice(120.0)
    xyz = catalogues.neyman_scott(n, 120.0, n // 50, 50.0, 3.0, n + periodic)
    edges = catalogues.linear_edges_lu(10.0, 15)
    ref = oracle.count_3pcf(xyz, box, periodic, edges)
    assert np.array_equal(gpu_3pcf(xyz, box, periodic, edges), ref)


def test_clustered_config_scaled_down():
    # the clustered workload's process and binning at 1/10 of its points in 1/10 of its volume
    w = configs.CLUSTERED_3PCF_D
    L = 500.0 / 10 ** (1 / 3)
    box = catalogues.box_lattice(L)
    xyz = catalogues.neyman_scott(20_000, L, 400, 50.0, 3.0, w.seed)
    ref = oracle.count_3pcf(xyz, box, 1, w.edges_lu)
    assert np.array_equal(gpu_3pcf(xyz, box, 1, w.edges_lu), ref)


def test_hub_rows_longer_than_the_table():
    # 2300 points within 0.45 r_max of each other: every pair is an edge, the
    # first hubs have > 2048 forward neighbours, so their rows run in chunks
    rng = np.random.default_rng(3)
    R = 40000
    v = rng.normal(size=(2300, 3))
    v *= (0.45 * R * rng.uniform(0, 1, size=(2300, 1)) ** (1 / 3)) / np.linalg.norm(v, axis=1, keepdims=True)
    xyz = (v + 100000).astype(np.int32)
    edges = [0, 9000, 21000, 33000, R]
    ref = oracle.count_3pcf(xyz, 300000, 0, edges)
    assert ref.sum() == 2300 * 2299 * 2298 // 6
    with gpu_graph(xyz, 300000, 0, edges) as g:
        assert g.max_degree == 2299
        assert np.array_equal(as_uint64(g.count_3pcf()), ref)


def test_two_cliques_rows_in_two_chunks():
    # two tight balls of a = 5200 and b = 3300 points, 30000 apart: pairs inside a
    # ball are closer than 9000 (bin 0), pairs across are 22000..38000 apart (bin 1).
    # Every pair is an edge, so the first hubs' forward rows hold more than 8192
    # keys and run in two chunks. Triangles: C(a,3) + C(b,3) of sides (0, 0, 0) and
    # C(a,2) b + C(b,2) a of sides (0, 1, 1).
    rng = np.random.default_rng(11)
    a, b = 5200, 3300

    def ball(m, centre):
        v = rng.normal(size=(m, 3))
        v *= 4000 * rng.uniform(0, 1, size=(m, 1)) ** (1 / 3) / np.linalg.norm(v, axis=1, keepdims=True)
        return (v + centre).astype(np.int32)

    xyz = np.concatenate([ball(a, 100000), ball(b, [130000, 100000, 100000])])
    xyz = xyz[rng.permutation(len(xyz))]
    edges = [0, 9000, 40000]
    with gpu_graph(xyz, 300000, 0, edges) as g:
        assert g.max_degree == a + b - 1
        hist = as_uint64(g.count_3pcf())
    c3 = lambda m: m * (m - 1) * (m - 2) // 6
    expect = {(0, 0, 0): c3(a) + c3(b), (0, 1, 1): a * (a - 1) // 2 * b + b * (b - 1) // 2 * a}
    cfg = fx.configs3(2)
    assert {cfg[k]: int(v) for k, v in enumerate(hist) if v} == expect


@pytest.mark.parametrize("nbins", [39, 40])
def test_most_bins_with_a_shared_histogram(nbins):
    # 39 and 40 bins: the largest histograms kept in shared memory. With short
    # rows the four-spoke walk is chosen, but its nb^3 table fits one block
    # only up to 39 bins; at 40 the count keeps the one-spoke walk
    box = catalogues.box_lattice(60.0)
    xyz = catalogues.uniform(3000, 60.0, 9)
    edges = catalogues.linear_edges_lu(12.0, nbins)
    ref = oracle.count_3pcf(xyz, box, 1, edges)
    assert ref.sum() > 0
    assert np.array_equal(gpu_3pcf(xyz, box, 1, edges), ref)


def test_hubs_whose_rows_wrap_the_box():
    # 400k uniform points in a periodic box, the input put in the graph's own
    # (cell) order, so that hub ranges mean the same to the oracle. The first
    # hubs lie in the first slab of cells; their forward neighbours include
    # points of the last slab across the periodic wrap, so their forward keys
    # span more than 2^18 ids and run as hash-table chunks. Hubs [0, 1000) are
    # counted against the oracle's hub loop over the same range (rows of those
    # hubs only, by brute force).
    import oracle as orc
    box = catalogues.box_lattice(1000.0)
    xyz = catalogues.uniform(400_000, 1000.0, 12)
    edges = catalogues.linear_edges_lu(30.0, 10)
    with gpu_graph(xyz, box, 1, edges) as g:
        perm = g.export_perm().cpu().numpy()
    xyz = np.ascontiguousarray(xyz[perm])
    hubs = 1000
    rows = [orc.row(xyz, box, 1, edges, i) for i in range(hubs)]
    spans = [int(r[r > i].max() - r[r > i].min() + 1) for i, (r, _) in enumerate(rows) if (r > i).sum() > 1]
    assert max(spans) > 1 << 18                       # hash-table chunks are exercised
    row_ptr = np.zeros(len(xyz) + 1, dtype=np.int64)
    row_ptr[1:hubs + 1] = np.cumsum([len(r) for r, _ in rows])
    row_ptr[hubs + 1:] = row_ptr[hubs]
    part = orc.Graph(row_ptr, np.concatenate([r for r, _ in rows]).astype(np.int32),
                     np.concatenate([b for _, b in rows]).astype(np.uint8))
    ref = orc.count_3pcf(xyz, box, 1, edges, g=part, hub_begin=0, hub_end=hubs)
    assert ref.sum() > 0
    with gpu_graph(xyz, box, 1, edges) as g:
        assert np.array_equal(g.export_perm().cpu().numpy(), np.arange(len(xyz)))
        assert np.array_equal(as_uint64(g.count_3pcf(0, hubs)), ref)


def test_many_bins_global_histogram():
    # C(62,3) = 37820 configurations: histogram too large for shared memory
    box = catalogues.box_lattice(60.0)
    xyz = catalogues.uniform(2500, 60.0, 8)
    edges = catalogues.linear_edges_lu(12.0, 60)
    ref = oracle.count_3pcf(xyz, box, 1, edges)
    assert np.array_equal(gpu_3pcf(xyz, box, 1, edges), ref)


def test_hub_ranges_sum_to_full():
    w = configs.TINY_3PCF
    xyz = w.points()
    full = oracle.count_3pcf(xyz, w.box_lu, 1, w.edges_lu)
    cuts = [0, 1, 2, 777, 1500, 1999, 2000]
    parts = gpu_3pcf(xyz, w.box_lu, 1, w.edges_lu, ranges=list(zip(cuts, cuts[1:])))
    assert np.array_equal(np.sum(parts, axis=0, dtype=np.uint64), full)
    assert gpu_3pcf(xyz, w.box_lu, 1, w.edges_lu, ranges=[(5, 5)])[0].sum() == 0


@pytest.mark.parametrize("periodic", [0, 1])
def test_invariances_on_the_gpu(periodic):
    box = catalogues.box_lattice(100.0)
    xyz = catalogues.neyman_scott(30_000, 100.0, 600, 50.0, 3.0, 123)
    edges = catalogues.linear_edges_lu(8.0, 10)
    base = gpu_3pcf(xyz, box, periodic, edges)
    assert base.sum() > 1e6
    perm = np.random.default_rng(2).permutation(len(xyz))
    assert np.array_equal(gpu_3pcf(xyz[perm], box, periodic, edges), base)
    assert np.array_equal(gpu_3pcf(mirror(xyz, box, periodic), box, periodic, edges), base)
    assert np.array_equal(gpu_3pcf(np.ascontiguousarray(xyz[:, [2, 0, 1]]), box, periodic, edges), base)
    if periodic:
        moved = ((xyz.astype(np.int64) + [51234, 7, 99999]) % box).astype(np.int32)
        assert np.array_equal(gpu_3pcf(moved, box, periodic, edges), base)


def test_host_buffer_entry_point():
    w = configs.TINY_3PCF
    xyz = w.points()
    ref = oracle.count_3pcf(xyz, w.box_lu, 1, w.edges_lu)
    assert np.array_equal(count_3pcf_from_host(xyz, w.box_lu, True, w.edges_lu), ref)


@pytest.mark.parametrize("n", [0, 1, 2, 3])
def test_tiny_inputs(n):
    xyz = np.full((n, 3), 500, dtype=np.int32)
    h = gpu_3pcf(xyz, 10000, 1, [0, 100, 200])
    assert int(h.sum()) == (1 if n == 3 else 0)
    if n == 3:
        assert h[0] == 1


_ABOVE_2_21 = {}


def _above_2_21_reference():
    """A uniform catalogue of 2,200,000 points (above 2^21, so the byte-map
    walks index their segment table relative to each chunk's first key, not by
    absolute segment) in a periodic box, in the graph's own order, with the
    oracle's unweighted and weighted counts over hubs [0, 500): rows of those
    hubs by brute force. The first hubs lie in the first cells, and their
    forward rows wrap the box, so they span more than 2^18 ids and run in
    several chunks."""
    if not _ABOVE_2_21:
        import oracle as orc
        box = catalogues.box_lattice(1000.0)
        xyz = catalogues.uniform(2_200_000, 1000.0, 31)
        edges = catalogues.linear_edges_lu(12.0, 5)
        with gpu_graph(xyz, box, 1, edges) as g:
            perm = g.export_perm().cpu().numpy()
        xyz = np.ascontiguousarray(xyz[perm])
        hubs = 500
        rows = [orc.row(xyz, box, 1, edges, i) for i in range(hubs)]
        spans = [int(r[r > i].max() - r[r > i].min() + 1) for i, (r, _) in enumerate(rows) if (r > i).sum() > 1]
        assert max(spans) > 1 << 18
        row_ptr = np.zeros(len(xyz) + 1, dtype=np.int64)
        row_ptr[1:hubs + 1] = np.cumsum([len(r) for r, _ in rows])
        row_ptr[hubs + 1:] = row_ptr[hubs]
        part = orc.Graph(row_ptr, np.concatenate([r for r, _ in rows]).astype(np.int32),
                         np.concatenate([b for _, b in rows]).astype(np.uint8))
        wt = np.random.default_rng(32).integers(-32767, 32768, size=len(xyz)).astype(np.int16)
        _ABOVE_2_21.update(xyz=xyz, box=box, edges=edges, hubs=hubs, wt=wt,
                           ref=orc.count_3pcf(xyz, box, 1, edges, g=part, hub_begin=0, hub_end=hubs),
                           ref_w=orc.count_3pcf_weighted(xyz, box, 1, edges, wt, g=part))
    return _ABOVE_2_21


def test_catalogue_above_2_21_points():
    import torch
    from cosmology_point_correlation_gb300 import as_int128
    r = _above_2_21_reference()
    assert r["ref"].sum() > 0
    with gpu_graph(r["xyz"], r["box"], 1, r["edges"]) as g:
        assert g.n > 1 << 21
        assert np.array_equal(g.export_perm().cpu().numpy(), np.arange(g.n))
        assert np.array_equal(as_uint64(g.count_3pcf(0, r["hubs"])), r["ref"])
        g.set_weights(torch.from_numpy(r["wt"]).cuda())
        assert as_int128(g.count_3pcf_weighted(0, r["hubs"])) == r["ref_w"]
