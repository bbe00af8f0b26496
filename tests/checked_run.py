"""Small cases through the checked build (run by tests/test_gpu_checked.py in a
process of its own with GRAMSCI_GB_LIBRARY set to libgramsci_gb_checked.so):
every result must equal the oracle's and no device check may fail (a failed
check would make the call raise GS_ERR_INTERNAL)."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from cosmology_point_correlation_gb300 import _lib, as_int128, as_uint64, catalogues, configs  # noqa: E402
from tests.gpu_util import gpu_graph, torch_dev  # noqa: E402


def main():
    lib = _lib.load()
    assert b"checked" in lib.gs_version(), lib.gs_version()
    torch, dev = torch_dev()
    cases = []                          # (points, box, periodic, edges); the last one is dense
    w = configs.TINY_3PCF
    cases.append((w.points(), w.box_lu, 1, w.edges_lu))
    for periodic in (0, 1):
        box = catalogues.box_lattice(120.0)
        cases.append((catalogues.neyman_scott(8000, 120.0, 160, 50.0, 3.0, 3 + periodic), box, periodic,
                      catalogues.linear_edges_lu(10.0, 15)))
    # 2300 points within 0.45 r_max of each other: every pair is an edge
    rng = np.random.default_rng(3)
    v = rng.normal(size=(2300, 3))
    v *= (0.45 * 40000 * rng.uniform(0, 1, size=(2300, 1)) ** (1 / 3)) / np.linalg.norm(v, axis=1, keepdims=True)
    cases.append(((v + 100000).astype(np.int32), 300000, 0, [0, 9000, 21000, 33000, 40000]))
    for c, (xyz, box, periodic, edges) in enumerate(cases):
        ref3 = oracle.count_3pcf(xyz, box, periodic, edges)
        for walk in ("map", "mapgroup", "warp", "group"):
            os.environ["GS_COUNT3_WALK"] = walk
            with gpu_graph(xyz, box, periodic, edges) as g:
                assert np.array_equal(as_uint64(g.count_3pcf()), ref3), walk
        os.environ.pop("GS_COUNT3_WALK")
        if c < 3:          # the dense case's parity count is O(n^4) for the oracle
            e, o = oracle.count_4pcf_parity(xyz, box, periodic, edges)
            with gpu_graph(xyz, box, periodic, edges) as g:
                ge, go = g.count_4pcf_parity()
                assert np.array_equal(as_uint64(ge), e) and np.array_equal(go.cpu().numpy(), o)
                hubs = np.arange(0, len(xyz), 7, dtype=np.int32)
                assert np.array_equal(as_uint64(g.count_3pcf_hubs(hubs)),
                                      oracle.count_3pcf_hubs(xyz, box, periodic, edges, hubs))
                wts = rng.integers(-32767, 32768, size=len(xyz)).astype(np.int16)
                g.set_weights(torch.from_numpy(wts).to(dev))
                assert as_int128(g.count_3pcf_weighted()) == oracle.count_3pcf_weighted(xyz, box, periodic, edges, wts)
    # two tight balls of a = 5200 and b = 3300 points whose pairs are all edges
    # (bin 0 inside a ball, bin 1 across): forward rows of more than 8192 keys
    # run in several chunks. Triangles in closed form: C(a,3) + C(b,3) of sides
    # (0, 0, 0), C(a,2) b + C(b,2) a of sides (0, 1, 1).
    a, b = 5200, 3300

    def ball(m, centre):
        u = rng.normal(size=(m, 3))
        u *= 4000 * rng.uniform(0, 1, size=(m, 1)) ** (1 / 3) / np.linalg.norm(u, axis=1, keepdims=True)
        return (u + centre).astype(np.int32)

    xyz = np.concatenate([ball(a, 100000), ball(b, [130000, 100000, 100000])])
    c3 = lambda m: m * (m - 1) * (m - 2) // 6                                   # noqa: E731
    for walk in ("map", "mapgroup", "warp", "group"):
        os.environ["GS_COUNT3_WALK"] = walk
        with gpu_graph(xyz, 300000, 0, [0, 9000, 40000]) as g:
            h = as_uint64(g.count_3pcf())
        assert int(h[0]) == c3(a) + c3(b) and int(h[2]) == a * (a - 1) // 2 * b + b * (b - 1) // 2 * a, walk
        assert int(h.sum()) == int(h[0]) + int(h[2]), walk
    os.environ.pop("GS_COUNT3_WALK")
    # windowed tiles with the byte-map walks
    xyz, box, periodic, edges = cases[2]
    from cosmology_point_correlation_gb300 import build_graph
    ref3 = oracle.count_3pcf(xyz, box, periodic, edges)
    with build_graph(torch.from_numpy(xyz).to(dev), box, periodic, edges, window_edges=60000) as g:
        assert g.windows()[0] > 2
        for walk in ("map", "mapgroup", "warp"):
            os.environ["GS_COUNT3_WALK"] = walk
            assert np.array_equal(as_uint64(g.count_3pcf()), ref3), walk
    print("checked build: all results equal the oracle, no device check failed")


if __name__ == "__main__":
    main()
