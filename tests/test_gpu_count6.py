"""Six-edge-bin 4pCF with parity channels on the GPU against the oracle
(GRAMSCI v2 §II.2 tetrahedra, §III.2 Eq.(3), §V.2 configurations)."""
import numpy as np
import pytest

import oracle
from cosmology_point_correlation_gb300 import as_uint64, catalogues, configs
from tests import fixtures as fx
from tests.gpu_util import gpu_graph, mirror

pytestmark = pytest.mark.gpu


def _gpu6(xyz, box, periodic, edges, ranges=None):
    with gpu_graph(xyz, box, periodic, edges) as g:
        if ranges is None:
            e, o = g.count_4pcf6()
            return as_uint64(e), o.cpu().numpy()
        out = [g.count_4pcf6(a, b) for a, b in ranges]
        return (np.sum([as_uint64(e) for e, _ in out], axis=0, dtype=np.uint64),
                np.sum([o.cpu().numpy() for _, o in out], axis=0))


@pytest.mark.parametrize("periodic", [0, 1])
@pytest.mark.parametrize("n,nb", [(3000, 4), (8000, 5)])
def test_matches_oracle(periodic, n, nb):
    L = 500.0 * (n / 200_000) ** (1 / 3)
    box = catalogues.box_lattice(L)
    xyz = catalogues.neyman_scott(n, L, max(1, n // 50), 50.0, 3.0, 21 + n + periodic)
    edges = catalogues.linear_edges_lu(20.0, nb)
    ref_e, ref_o = oracle.count_4pcf6(xyz, box, periodic, edges)
    assert ref_e.sum() > 10_000 and np.abs(ref_o).sum() > 0
    e, o = _gpu6(xyz, box, periodic, edges)
    assert np.array_equal(e, ref_e) and np.array_equal(o, ref_o)


def test_fixture_shapes():
    shapes = {s["name"]: s for s in fx.tetrahedron_shapes()}
    box = 1_000_000
    for name in ("T", "T_mirror", "T_relabel", "R", "P"):
        xyz = (shapes[name]["vertices"] + 500_000).astype(np.int32)
        ref_e, ref_o = oracle.count_4pcf6(xyz, box, 0, fx.TETRA_EDGES)
        e, o = _gpu6(xyz, box, 0, fx.TETRA_EDGES)
        assert np.array_equal(e, ref_e) and np.array_equal(o, ref_o), name
    k = oracle.config_index6(4, (0, 1, 2, 2, 2, 3))
    e, o = _gpu6((shapes["T"]["vertices"] + 500_000).astype(np.int32), box, 0, fx.TETRA_EDGES)
    assert e[k] == 1 and o[k] == 1


@pytest.mark.parametrize("m", [100, 200, 300])
def test_hubs_of_each_shared_memory_size(m):
    # a hub (input index 0) at the corner of cell 0 with m neighbours on an
    # octant shell of radius 0.45..0.9 r_max, all in cell 0, so all m are
    # forward neighbours: the 128-slot kernel, the 256-slot kernel and the
    # global-scratch path
    rng = np.random.default_rng(8)
    R = 20000
    v = np.abs(rng.normal(size=(m, 3)))
    v *= (0.9 * R * (0.5 + 0.5 * rng.uniform(size=(m, 1)))) / np.linalg.norm(v, axis=1, keepdims=True)
    xyz = (np.vstack([[[0, 0, 0]], np.rint(v)]) + 100).astype(np.int32)
    edges = [0, 8000, 12000, 16000, R]
    ref_e, ref_o = oracle.count_4pcf6(xyz, 80000, 0, edges)
    assert ref_e.sum() > 1000
    with gpu_graph(xyz, 80000, 0, edges) as g:
        assert g.stats()["max_forward"] == m
        e, o = g.count_4pcf6()
        assert np.array_equal(as_uint64(e), ref_e) and np.array_equal(o.cpu().numpy(), ref_o)


def test_parity_catalogue_four_bins_full_size():
    w = configs.PARITY_4PCF
    xyz = w.points()
    edges = catalogues.linear_edges_lu(w.r_max_mpc, 4)
    e, o = _gpu6(xyz, w.box_lu, True, edges)
    assert len(e) == 276 and e.sum() > 0
    n = len(xyz)
    e2, o2 = _gpu6(xyz, w.box_lu, True, edges, ranges=[(0, n // 3), (n // 3, n)])
    assert np.array_equal(e2, e) and np.array_equal(o2, o)
    e3, o3 = _gpu6(mirror(xyz, w.box_lu, True), w.box_lu, True, edges)
    assert np.array_equal(e3, e) and np.array_equal(o3, -o)


# ---------------------------------------------------------------- weighted (§II.1 signed weights)

def _gpu6w(xyz, box, periodic, edges, w, ranges=None):
    from cosmology_point_correlation_gb300 import as_int128
    from tests.gpu_util import torch_dev
    torch, dev = torch_dev()
    with gpu_graph(xyz, box, periodic, edges) as g:
        g.set_weights(torch.from_numpy(np.ascontiguousarray(w, dtype=np.int16)).to(dev))
        if ranges is None:
            e, o = g.count_4pcf6_weighted()
            return as_int128(e), as_int128(o)
        parts = [g.count_4pcf6_weighted(a, b) for a, b in ranges]
        return ([sum(c) for c in zip(*[as_int128(e) for e, _ in parts])],
                [sum(c) for c in zip(*[as_int128(o) for _, o in parts])])


def _weights(n, seed):
    return np.random.default_rng(seed).integers(-32767, 32768, size=n).astype(np.int16)


@pytest.mark.parametrize("periodic", [0, 1])
@pytest.mark.parametrize("n,nb", [(3000, 4), (8000, 5), (3000, 7)])
def test_weighted_matches_oracle(periodic, n, nb):
    # 4 and 5 bins: block sums in shared memory; 7 bins (5475 configurations):
    # straight into the global sums
    L = 500.0 * (n / 200_000) ** (1 / 3)
    box = catalogues.box_lattice(L)
    xyz = catalogues.neyman_scott(n, L, max(1, n // 50), 50.0, 3.0, 21 + n + periodic)
    edges = catalogues.linear_edges_lu(20.0, nb)
    w = _weights(n, n + nb)
    ref = oracle.count_4pcf6_weighted(xyz, box, periodic, edges, w)
    assert any(ref[1])
    assert _gpu6w(xyz, box, periodic, edges, w) == ref


def test_weighted_large_hub_and_extreme_weights():
    rng = np.random.default_rng(8)
    R = 20000
    v = rng.normal(size=(300, 3))
    v *= (0.9 * R * (0.5 + 0.5 * rng.uniform(size=(300, 1)))) / np.linalg.norm(v, axis=1, keepdims=True)
    xyz = (np.vstack([[[0, 0, 0]], np.rint(v)]) + 25000).astype(np.int32)
    edges = [0, 8000, 12000, 16000, R]
    w = _weights(len(xyz), 3)
    assert _gpu6w(xyz, 50000, 0, edges, w) == oracle.count_4pcf6_weighted(xyz, 50000, 0, edges, w)
    # constant -32767: every term is (-32767)^4 ~ 2^60, sums leave int64
    c = np.full(len(xyz), -32767, np.int16)
    e, o = oracle.count_4pcf6(xyz, 50000, 0, edges)
    ge, go = _gpu6w(xyz, 50000, 0, edges, c)
    assert ge == [int(x) * 32767 ** 4 for x in e] and go == [int(x) * 32767 ** 4 for x in o]
    assert max(ge) > 1 << 63


def test_weighted_parity_catalogue_unit_weights_and_ranges():
    w = configs.PARITY_4PCF
    xyz = w.points()
    edges = catalogues.linear_edges_lu(w.r_max_mpc, 4)
    e, o = _gpu6(xyz, w.box_lu, True, edges)
    one = np.ones(len(xyz), np.int16)
    assert _gpu6w(xyz, w.box_lu, True, edges, one) == ([int(x) for x in e], [int(x) for x in o])
    n = len(xyz)
    wt = _weights(n, 77)
    full = _gpu6w(xyz, w.box_lu, True, edges, wt)
    assert _gpu6w(xyz, w.box_lu, True, edges, wt, ranges=[(0, n // 3), (n // 3, n)]) == full
    # mirror image: even unchanged, odd negated (weights travel with the points)
    me, mo = _gpu6w(mirror(xyz, w.box_lu, True), w.box_lu, True, edges, wt)
    assert me == full[0] and mo == [-x for x in full[1]]
