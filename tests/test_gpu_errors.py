"""Host-side argument errors: each returns its status with a message and
leaves no graph behind. Nothing here faults a device."""
import ctypes

import numpy as np
import pytest

from cosmology_point_correlation_gb300 import GramsciError, _lib, build_graph, catalogues
from tests.gpu_util import gpu_graph, torch_dev

pytestmark = pytest.mark.gpu


def _coords(n=100, box=10000, seed=0):
    torch, dev = torch_dev()
    return torch.from_numpy(catalogues.uniform(n, box / 1024, seed)).to(dev)


@pytest.mark.parametrize("edges,periodic,box,msg", [
    ([0], 1, 10000, "at least two"),
    ([0, 100, 100], 1, 10000, "strictly increasing"),
    ([-5, 100], 1, 10000, "edges_lu[0]"),
    ([0, 6000], 1, 10000, "2*r_max_lu"),
    (list(range(0, 257 * 10, 10)), 0, 10000, "nbins"),
])
def test_bad_build_arguments(edges, periodic, box, msg):
    with pytest.raises((GramsciError, ValueError), match=msg.replace("*", r"\*").replace("[", r"\[")):
        build_graph(_coords(box=box), box, periodic, edges)


def test_coordinate_out_of_range_is_reported():
    torch, dev = torch_dev()
    xyz = catalogues.uniform(1000, 10000 / 1024, 1)
    xyz[500, 1] = 10000                      # == box: outside [0, box)
    with pytest.raises(GramsciError) as e:
        build_graph(torch.from_numpy(xyz).to(dev), 10000, 1, [0, 500, 1000])
    assert e.value.status == _lib.GS_ERR_ARG and "outside" in str(e.value)
    xyz[500, 1] = -1
    with pytest.raises(GramsciError):
        build_graph(torch.from_numpy(xyz).to(dev), 10000, 0, [0, 500, 1000])


def test_box_limits():
    lib = _lib.load()
    h = ctypes.c_void_p()
    e = np.array([0, 10], dtype=np.int64)
    c = _coords()
    assert lib.gs_build_graph(ctypes.c_void_p(c.data_ptr()), 100, (1 << 30) + 1, 0, 10,
                              e.ctypes.data_as(ctypes.c_void_p), 1, None, ctypes.byref(h)) == _lib.GS_ERR_ARG
    assert not h.value
    assert lib.gs_build_graph(ctypes.c_void_p(c.data_ptr()), -1, 10000, 0, 10,
                              e.ctypes.data_as(ctypes.c_void_p), 1, None, ctypes.byref(h)) == _lib.GS_ERR_ARG
    assert lib.gs_build_graph(ctypes.c_void_p(c.data_ptr()), 100, 10000, 0, 11,
                              e.ctypes.data_as(ctypes.c_void_p), 1, None, ctypes.byref(h)) == _lib.GS_ERR_ARG
    assert b"r_max_lu" in lib.gs_last_error()


def test_bad_count_arguments():
    torch, dev = torch_dev()
    xyz = catalogues.uniform(500, 10000 / 1024, 2)
    with gpu_graph(xyz, 10000, 1, [0, 1000, 2000, 3000]) as g:
        with pytest.raises(GramsciError, match="hub range"):
            g.count_3pcf(0, 501)
        with pytest.raises(GramsciError, match="hub range"):
            g.count_3pcf(10, 5)
        with pytest.raises(GramsciError, match="hub range"):
            g.count_4pcf_parity(-1, 5)
        lib = _lib.load()
        assert lib.gs_count_3pcf(g._h, None, 0, 500, None) == _lib.GS_ERR_ARG


def test_parity_needs_exact_volume_range():
    xyz = catalogues.uniform(200, 8192.0, 3)
    box = catalogues.box_lattice(8192.0)          # 2^23 >= 2 r_max
    with gpu_graph(xyz, box, 1, [0, 1 << 19, 1 << 20, 3 << 20]) as g:
        with pytest.raises(GramsciError, match="2\\^20"):
            g.count_4pcf_parity()
        g.count_3pcf()                         # the 3pCF has no such limit


def test_graph_of_another_device_is_refused():
    # every count and export checks that the current device is the graph's own
    # (a graph's pointers are meaningless on another device). With one GPU the
    # test makes the recorded device differ instead of switching devices.
    torch, dev = torch_dev()
    xyz = catalogues.uniform(300, 10000 / 1024, 4)
    lib = _lib.load()
    with gpu_graph(xyz, 10000, 1, [0, 1000, 2000, 3000]) as g:
        rec = ctypes.cast(g._h, ctypes.POINTER(ctypes.c_int))   # the handle's first field is its device
        own = rec[0]
        hist = torch.zeros(20, dtype=torch.int64, device=dev)
        rec[0] = own + 1
        try:
            for call in (lambda: lib.gs_count_3pcf(g._h, ctypes.c_void_p(hist.data_ptr()), 0, 300, None),
                         lambda: lib.gs_count_4pcf_parity(g._h, ctypes.c_void_p(hist.data_ptr()),
                                                          ctypes.c_void_p(hist.data_ptr()), 0, 300, None),
                         lambda: lib.gs_count_2pcf(g._h, ctypes.c_void_p(hist.data_ptr()), None),
                         lambda: lib.gs_graph_hub_work(g._h, None, ctypes.c_void_p(hist.data_ptr()), None)):
                assert call() == _lib.GS_ERR_ARG
                assert b"device" in lib.gs_last_error()
        finally:
            rec[0] = own
        assert lib.gs_count_3pcf(g._h, ctypes.c_void_p(hist.data_ptr()), 0, 300, None) == _lib.GS_OK
