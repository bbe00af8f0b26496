"""Weighted 2pCF and 3pCF on the GPU equal the oracle exactly (GRAMSCI v2
§II.1, §III.3: counts with signed data-minus-random weights; here int16
fixed-point weights, sums as exact 128-bit integers)."""
import numpy as np
import pytest

import oracle
from cosmology_point_correlation_gb300 import GramsciError, as_int128, as_uint64, catalogues, configs
from tests.gpu_util import gpu_graph, mirror, torch_dev

pytestmark = pytest.mark.gpu


def _weights(n, seed, lo=-32767, hi=32767):
    return np.random.default_rng(seed).integers(lo, hi + 1, size=n).astype(np.int16)


def _set(g, w):
    torch, dev = torch_dev()
    g.set_weights(torch.from_numpy(w).to(dev))


def _clustered(n, seed, periodic=1):
    box = catalogues.box_lattice(120.0)
    xyz = catalogues.neyman_scott(n, 120.0, n // 50, 50.0, 3.0, seed + periodic)
    return xyz, box, catalogues.linear_edges_lu(10.0, 15)


def test_unit_weights_equal_the_counts():
    w = configs.TINY_3PCF
    xyz = w.points()
    with gpu_graph(xyz, w.box_lu, 1, w.edges_lu) as g:
        _set(g, np.ones(len(xyz), np.int16))
        assert as_int128(g.count_2pcf_weighted()) == [int(v) for v in as_uint64(g.count_2pcf())]
        assert as_int128(g.count_3pcf_weighted()) == [int(v) for v in as_uint64(g.count_3pcf())]
        assert as_int128(g.count_2pcf_weighted()) == [int(v) for v in as_uint64(g.count_2pcf())]


@pytest.mark.parametrize("walk", ["map", "warp"])
@pytest.mark.parametrize("periodic", [0, 1])
@pytest.mark.parametrize("n", [5_000, 20_011])
def test_random_weights_clustered(periodic, n, walk, monkeypatch):
    # the byte-map walk (default) and the bitmap walk of the weighted count
    monkeypatch.setenv("GS_COUNT3_WALK", walk)
    xyz, box, edges = _clustered(n, n, periodic)
    wt = _weights(n, n + 7)
    with gpu_graph(xyz, box, periodic, edges) as g:
        _set(g, wt)
        assert as_int128(g.count_2pcf_weighted()) == oracle.count_2pcf_weighted(xyz, box, periodic, edges, wt)
        assert as_int128(g.count_3pcf_weighted()) == oracle.count_3pcf_weighted(xyz, box, periodic, edges, wt)


def test_constant_negative_weights_sign_extend():
    # every weight -32767: each triangle adds -(32767^3), each pair -(-32767)^2
    w = configs.TINY_3PCF
    xyz = w.points()
    wt = np.full(len(xyz), -32767, np.int16)
    with gpu_graph(xyz, w.box_lu, 1, w.edges_lu) as g:
        _set(g, wt)
        h3 = as_int128(g.count_3pcf_weighted())
        h2 = as_int128(g.count_2pcf_weighted())
    assert h3 == [-int(v) * 32767 ** 3 for v in oracle.count_3pcf(xyz, w.box_lu, 1, w.edges_lu)]
    assert h2 == [int(v) * 32767 ** 2 for v in oracle.count_2pcf(xyz, w.box_lu, 1, w.edges_lu)]


def test_hub_ranges_add_up():
    xyz, box, edges = _clustered(20_011, 3)
    wt = _weights(len(xyz), 11)
    with gpu_graph(xyz, box, 1, edges) as g:
        _set(g, wt)
        full = as_int128(g.count_3pcf_weighted())
        cuts = [0, 1, 777, 12_345, len(xyz)]
        parts = [as_int128(g.count_3pcf_weighted(a, b)) for a, b in zip(cuts[:-1], cuts[1:])]
        assert [sum(col) for col in zip(*parts)] == full
        assert as_int128(g.count_3pcf_weighted(5, 5)) == [0] * len(full)


def test_hub_rows_longer_than_the_table():
    # a clique of 2300 points: the first hubs' forward rows run in two chunks
    rng = np.random.default_rng(3)
    R = 40000
    v = rng.normal(size=(2300, 3))
    v *= (0.45 * R * rng.uniform(0, 1, size=(2300, 1)) ** (1 / 3)) / np.linalg.norm(v, axis=1, keepdims=True)
    xyz = (v + 100000).astype(np.int32)
    edges = [0, 9000, 21000, 33000, R]
    wt = _weights(len(xyz), 5)
    with gpu_graph(xyz, 300000, 0, edges) as g:
        assert g.stats()["max_forward"] > 2048
        _set(g, wt)
        assert as_int128(g.count_3pcf_weighted()) == oracle.count_3pcf_weighted(xyz, 300000, 0, edges, wt)
        assert as_int128(g.count_2pcf_weighted()) == oracle.count_2pcf_weighted(xyz, 300000, 0, edges, wt)
        # constant -32767: ~1e8 triangles per configuration times -2^45 leaves
        # int64, so the carries into the high word are exercised
        _set(g, np.full(len(xyz), -32767, np.int16))
        h3 = as_int128(g.count_3pcf_weighted())
    ref = [-int(v) * 32767 ** 3 for v in oracle.count_3pcf(xyz, 300000, 0, edges)]
    assert min(ref) < -(1 << 63)
    assert h3 == ref


@pytest.mark.parametrize("walk", ["map", "warp"])
def test_two_cliques_rows_in_two_chunks(walk, monkeypatch):
    # Two tight balls of a = 5200 and b = 3300 points 30000 apart, every pair an
    # edge (bin 0 inside a ball, bin 1 across): the first hubs' forward rows
    # hold more than 8192 keys and run in two chunks. With weights w, the sums
    # are elementary symmetric polynomials of each ball's weights, computed
    # exactly from power sums (Newton's identities): (0, 0, 0) gets
    # e3(A) + e3(B), (0, 1, 1) gets e2(A) e1(B) + e2(B) e1(A).
    monkeypatch.setenv("GS_COUNT3_WALK", walk)
    rng = np.random.default_rng(11)
    a, b = 5200, 3300

    def ball(m, centre):
        v = rng.normal(size=(m, 3))
        v *= 4000 * rng.uniform(0, 1, size=(m, 1)) ** (1 / 3) / np.linalg.norm(v, axis=1, keepdims=True)
        return (v + centre).astype(np.int32)

    xyz = np.concatenate([ball(a, 100000), ball(b, [130000, 100000, 100000])])
    wt = _weights(a + b, 12)
    order = rng.permutation(a + b)
    edges = [0, 9000, 40000]

    def e123(w):
        p1, p2, p3 = (sum(int(x) ** k for x in w) for k in (1, 2, 3))
        return p1, (p1 * p1 - p2) // 2, (p1 ** 3 - 3 * p1 * p2 + 2 * p3) // 6

    ea, eb = e123(wt[:a]), e123(wt[a:])
    with gpu_graph(xyz[order], 300000, 0, edges) as g:
        assert g.max_degree == a + b - 1
        _set(g, wt[order])
        sums = as_int128(g.count_3pcf_weighted())
    # configurations of 2 bins in lexicographic order: (0,0,0) (0,0,1) (0,1,1) (1,1,1)
    assert sums == [ea[2] + eb[2], 0, ea[1] * eb[0] + eb[1] * ea[0], 0]


@pytest.mark.parametrize("nb", [1, 32, 33, 40])
def test_bin_counts(nb):
    # 40 bins: 11480 configurations (one block per SM); above 32 bins the
    # 2pCF takes its shared 128-bit path
    xyz, box, _ = _clustered(8_000, 21 + nb)
    edges = catalogues.linear_edges_lu(10.0, nb)
    wt = _weights(len(xyz), 22 + nb)
    with gpu_graph(xyz, box, 1, edges) as g:
        _set(g, wt)
        assert as_int128(g.count_3pcf_weighted()) == oracle.count_3pcf_weighted(xyz, box, 1, edges, wt)
        assert as_int128(g.count_2pcf_weighted()) == oracle.count_2pcf_weighted(xyz, box, 1, edges, wt)


def test_data_minus_random_weights_and_mirror():
    # data +a, randoms -b: the pair sum is a^2 DD - 2ab DR + b^2 RR (§III.3)
    box = catalogues.box_lattice(120.0)
    d = catalogues.neyman_scott(6_000, 120.0, 120, 50.0, 3.0, 31)
    r = catalogues.uniform(9_000, 120.0, 32)
    xyz = np.concatenate([d, r])
    wt = np.concatenate([np.full(len(d), 300, np.int16), np.full(len(r), -200, np.int16)])
    edges = catalogues.linear_edges_lu(10.0, 15)
    with gpu_graph(xyz, box, 1, edges) as g:
        _set(g, wt)
        s2 = as_int128(g.count_2pcf_weighted())
        s3 = as_int128(g.count_3pcf_weighted())
    assert s2 == oracle.count_2pcf_weighted(xyz, box, 1, edges, wt)
    assert s3 == oracle.count_3pcf_weighted(xyz, box, 1, edges, wt)
    with gpu_graph(mirror(xyz, box, 1), box, 1, edges) as g:
        _set(g, wt)
        assert as_int128(g.count_2pcf_weighted()) == s2
        assert as_int128(g.count_3pcf_weighted()) == s3


def test_errors():
    torch, dev = torch_dev()
    w = configs.TINY_3PCF
    xyz = w.points()
    with gpu_graph(xyz, w.box_lu, 1, w.edges_lu) as g:
        with pytest.raises(GramsciError, match="no weights"):
            g.count_3pcf_weighted()
        with pytest.raises(GramsciError, match="no weights"):
            g.count_2pcf_weighted()
        with pytest.raises(TypeError):
            g.set_weights(torch.ones(len(xyz), dtype=torch.int32, device=dev))
        with pytest.raises(ValueError):
            g.set_weights(torch.ones(len(xyz) - 1, dtype=torch.int16, device=dev))
        _set(g, np.ones(len(xyz), np.int16))
        with pytest.raises(GramsciError):
            g.count_3pcf_weighted(0, len(xyz) + 1)
    with gpu_graph(xyz, w.box_lu, 1, catalogues.linear_edges_lu(20.0, 41)) as g:
        _set(g, np.ones(len(xyz), np.int16))
        with pytest.raises(GramsciError, match="at most 40"):
            g.count_3pcf_weighted()


@pytest.mark.slow
def test_bao_workload_unit_weights():
    # the 2M-point, 30-bin open-box workload (4960 configurations): unit
    # weights reproduce the triangle and pair counts
    w = configs.BAO_3PCF
    xyz = w.points()
    with gpu_graph(xyz, w.box_lu, w.periodic, w.edges_lu) as g:
        _set(g, np.ones(len(xyz), np.int16))
        assert as_int128(g.count_3pcf_weighted()) == [int(v) for v in as_uint64(g.count_3pcf())]
        assert as_int128(g.count_2pcf_weighted()) == [int(v) for v in as_uint64(g.count_2pcf())]
