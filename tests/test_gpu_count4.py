"""Parity-4pCF histograms on the GPU equal the oracle bit for bit
(GRAMSCI v2 §III.1.1, §III.2 Eq.(3), degenerate rule; §IV.9 injection)."""
import numpy as np
import pytest

import oracle
from cosmology_point_correlation_gb300 import catalogues, configs, count_4pcf_parity_from_host
from tests import fixtures as fx
from tests.gpu_util import gpu_4pcf, gpu_graph, mirror

pytestmark = pytest.mark.gpu


def _check(xyz, box, periodic, edges):
    ref_e, ref_o = oracle.count_4pcf_parity(xyz, box, periodic, edges)
    e, o = gpu_4pcf(xyz, box, periodic, edges)
    assert np.array_equal(e, ref_e)
    assert np.array_equal(o, ref_o)
    return ref_e, ref_o


@pytest.mark.parametrize("periodic", [0, 1])
@pytest.mark.parametrize("n", [4_000, 20_003])
def test_parity_workload_scaled_down(periodic, n):
    # the parity workload's process (sigma 3, 50 per cluster) and 8 bins of 2.5 Mpc
    w = configs.PARITY_4PCF
    L = 500.0 * (n / w.n) ** (1 / 3)
    box = catalogues.box_lattice(L)
    xyz = catalogues.neyman_scott(n, L, max(1, n // 50), 50.0, 3.0, w.seed + n)
    ref_e, ref_o = _check(xyz, box, periodic, w.edges_lu)
    assert ref_e.sum() > 10_000 and np.abs(ref_o).sum() > 0


def test_shapes_from_fixtures():
    shapes = {s["name"]: s for s in fx.tetrahedron_shapes()}
    box = 1_000_000
    cfg = fx.configs4(4)
    for name, s in shapes.items():
        xyz = (s["vertices"] + 500_000).astype(np.int32)
        e, o = gpu_4pcf(xyz, box, 0, fx.TETRA_EDGES)
        ee = np.zeros(len(cfg), dtype=np.uint64)
        oo = np.zeros(len(cfg), dtype=np.int64)
        for _, bins, ev, od in s["hubs"]:
            ee[cfg.index(bins)] += ev
            oo[cfg.index(bins)] += od
        assert np.array_equal(e, ee) and np.array_equal(o, oo), name


def test_chiral_injection():
    shapes = {s["name"]: s for s in fx.tetrahedron_shapes()}
    left, right = shapes["T"]["vertices"], shapes["T_mirror"]["vertices"]
    box = 1_000_000
    pts = []
    n_left, n_right = 37, 14
    for c in range(n_left + n_right):
        origin = np.array([5000 + 12000 * (c % 40), 5000 + 12000 * (c // 40), 5000])
        pts.extend((left if c < n_left else right) + origin)
    xyz = np.array(pts, dtype=np.int32)
    e, o = gpu_4pcf(xyz, box, 0, fx.TETRA_EDGES)
    # per unit: (0,1,2) and (1,2,3) once each, odd +1 (left) / -1 (right)
    cfg = fx.configs4(4)
    for bins in [(0, 1, 2), (1, 2, 3)]:
        k = cfg.index(bins)
        assert e[k] == n_left + n_right and o[k] == n_left - n_right


def test_hub_of_degree_above_shared_limit():
    # a hub with 520 neighbours (uniform in a ball of 0.98 r_max) runs in the
    # scratch-memory kernel; the others stay in shared memory
    rng = np.random.default_rng(11)
    R = 20000
    v = rng.normal(size=(520, 3))
    v *= (0.98 * R * rng.uniform(0, 1, size=(520, 1)) ** (1 / 3)) / np.linalg.norm(v, axis=1, keepdims=True)
    xyz = np.vstack([[[0, 0, 0]], np.rint(v)]).astype(np.int64) + 100000
    xyz = xyz.astype(np.int32)
    edges = [0, 5000, 9000, 12500, 16000, 18000, R]
    with gpu_graph(xyz, 500000, 0, edges) as g:
        assert g.max_degree >= 520
    _check(xyz, 500000, 0, edges)


def test_many_bins_global_histogram():
    # C(40,3) = 9880 configurations: histograms in global memory
    box = catalogues.box_lattice(50.0)
    xyz = catalogues.neyman_scott(3000, 50.0, 60, 50.0, 2.0, 17)
    _check(xyz, box, 1, catalogues.linear_edges_lu(10.0, 40))


def test_hub_ranges_sum_to_full():
    box = catalogues.box_lattice(60.0)
    xyz = catalogues.neyman_scott(5000, 60.0, 100, 50.0, 3.0, 5)
    edges = catalogues.linear_edges_lu(10.0, 8)
    ref_e, ref_o = oracle.count_4pcf_parity(xyz, box, 1, edges)
    cuts = [0, 3, 1000, 2500, 4999, 5000]
    parts = gpu_4pcf(xyz, box, 1, edges, ranges=list(zip(cuts, cuts[1:])))
    assert np.array_equal(np.sum([p[0] for p in parts], axis=0, dtype=np.uint64), ref_e)
    assert np.array_equal(np.sum([p[1] for p in parts], axis=0), ref_o)


@pytest.mark.parametrize("periodic", [0, 1])
def test_mirror_and_rotation_on_the_gpu(periodic):
    box = catalogues.box_lattice(80.0)
    xyz = catalogues.neyman_scott(12_000, 80.0, 240, 50.0, 3.0, 31)
    edges = catalogues.linear_edges_lu(10.0, 8)
    e, o = gpu_4pcf(xyz, box, periodic, edges)
    assert np.abs(o).sum() > 0
    e2, o2 = gpu_4pcf(mirror(xyz, box, periodic), box, periodic, edges)
    assert np.array_equal(e2, e) and np.array_equal(o2, -o)
    e3, o3 = gpu_4pcf(np.ascontiguousarray(xyz[:, [1, 2, 0]]), box, periodic, edges)
    assert np.array_equal(e3, e) and np.array_equal(o3, o)
    perm = np.random.default_rng(4).permutation(len(xyz))
    e4, o4 = gpu_4pcf(xyz[perm], box, periodic, edges)
    assert np.array_equal(e4, e) and np.array_equal(o4, o)


def test_host_buffer_entry_point():
    box = catalogues.box_lattice(60.0)
    xyz = catalogues.neyman_scott(5000, 60.0, 100, 50.0, 3.0, 6)
    edges = catalogues.linear_edges_lu(10.0, 8)
    ref_e, ref_o = oracle.count_4pcf_parity(xyz, box, 1, edges)
    e, o = count_4pcf_parity_from_host(xyz, box, True, edges)
    assert np.array_equal(e, ref_e) and np.array_equal(o, ref_o)


def test_fewer_than_three_bins_write_nothing():
    xyz = catalogues.uniform(100, 20.0, 1)
    e, o = gpu_4pcf(xyz, catalogues.box_lattice(20.0), 1, [0, 1000, 4000])
    assert len(e) == 0 and len(o) == 0
