"""Allocation failures, injected on the host (GS_FAULT=alloc:N makes the N-th
allocation of a call fail without allocating): every call that allocates
returns GS_ERR_NOMEM at each of its allocation sites, leaves its outputs
unwritten, and frees what it had allocated. No device fault is involved:
the failing allocation is never attempted.

The paper's counterpart is the automatic switch to tiled (windowed) operation
when device memory runs short (GRAMSCI v2 §III.5.3); here the failure paths
of every allocation site are exercised directly.
"""
import ctypes

import numpy as np
import pytest

from cosmology_point_correlation_gb300 import _lib, catalogues
from tests.gpu_util import gpu_graph, torch_dev

pytestmark = pytest.mark.gpu

SENTINEL = 0x5A5A5A5A5A5A5A5A


def _star(deg=700, R=20000, seed=23, background=0):
    # one hub whose neighbours fill a ball of 0.98 r_max: rows longer than the
    # shared-memory kernels take, so the large-hub workspaces are allocated;
    # uniform background points spread the graph over many cells (windows)
    rng = np.random.default_rng(seed)
    v = rng.normal(size=(deg, 3))
    v *= (0.98 * R * rng.uniform(0, 1, size=(deg, 1)) ** (1 / 3)) / np.linalg.norm(v, axis=1, keepdims=True)
    xyz = np.vstack([[[0, 0, 0]], np.rint(v)]) + 100000
    if background:
        xyz = np.vstack([xyz, rng.integers(0, 500000, size=(background, 3))])
    return xyz.astype(np.int32), 500000, 0, np.array([0, 5000, 9000, 12500, 16000, 18000, R], dtype=np.int64)


def _free_bytes(torch):
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0]


def _sweep(call, outputs, torch, monkeypatch, max_sites=64):
    """Fail allocation 1, 2, ... of `call` until it succeeds; returns the number
    of allocation sites met. `outputs` are tensors that must stay unwritten."""
    monkeypatch.delenv("GS_FAULT", raising=False)
    assert call() == _lib.GS_OK                       # warm: lazy module loads, tables built on first use
    for n in range(1, max_sites + 1):
        for t in outputs:
            t.fill_(SENTINEL)
        before = _free_bytes(torch)
        monkeypatch.setenv("GS_FAULT", f"alloc:{n}")
        status = call()
        monkeypatch.delenv("GS_FAULT")
        after = _free_bytes(torch)
        if status == _lib.GS_OK:
            return n - 1
        assert status == _lib.GS_ERR_NOMEM, (n, status, _lib.load().gs_last_error())
        assert _lib.load().gs_last_error()
        for t in outputs:
            assert bool((t == SENTINEL).all()), f"allocation {n}: an output was written"
        assert after == before, f"allocation {n}: {before - after} bytes not freed"
    raise AssertionError("more allocation sites than expected")


def test_build_graph_every_allocation(monkeypatch):
    torch, dev = torch_dev()
    lib = _lib.load()
    box = catalogues.box_lattice(60.0)
    xyz = torch.from_numpy(catalogues.uniform(3000, 60.0, 2)).to(dev)
    edges = catalogues.linear_edges_lu(10.0, 5)
    for window in (0, 20000):
        def call():
            h = ctypes.c_void_p()
            args = (ctypes.c_void_p(xyz.data_ptr()), 3000, box, 1, int(edges[-1]),
                    edges.ctypes.data_as(ctypes.c_void_p), len(edges) - 1)
            if window:
                s = lib.gs_build_graph_windowed(*args, window, None, ctypes.byref(h))
            else:
                s = lib.gs_build_graph(*args, None, ctypes.byref(h))
            if s == _lib.GS_OK:
                lib.gs_graph_free(h)
            else:
                assert not h.value                    # no graph handed out
            return s
        assert _sweep(call, [], torch, monkeypatch) >= 10


@pytest.mark.parametrize("windowed", [0, 1])
def test_counts_every_allocation(windowed, monkeypatch):
    torch, dev = torch_dev()
    lib = _lib.load()
    xyz, box, periodic, edges = _star(background=20000 if windowed else 0)
    nb = len(edges) - 1
    g = gpu_graph(xyz, box, periodic, edges) if not windowed else None
    if windowed:
        from cosmology_point_correlation_gb300 import build_graph
        g = build_graph(torch.from_numpy(xyz).to(dev), box, periodic, edges, window_edges=60000)
        assert g.windows()[0] > 1
    with g:
        st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        g.set_weights(torch.from_numpy(np.random.default_rng(1).integers(-900, 900, size=len(xyz))
                                       .astype(np.int16)).to(dev))
        n3, n4 = nb * (nb + 1) * (nb + 2) // 6, nb * (nb - 1) * (nb - 2) // 6
        n6 = lib.gs_config_count_4pcf6(nb)
        h3 = torch.empty(2 * n3, dtype=torch.int64, device=dev)
        ev = torch.empty(2 * n6, dtype=torch.int64, device=dev)
        od = torch.empty(2 * n6, dtype=torch.int64, device=dev)
        p = lambda t: ctypes.c_void_p(t.data_ptr())        # noqa: E731
        calls = {
            "3pcf_weighted": (lambda: lib.gs_count_3pcf_weighted(g._h, p(h3), 0, len(xyz), st), [h3]),
            "4pcf_parity": (lambda: lib.gs_count_4pcf_parity(g._h, p(ev), p(od), 0, len(xyz), st), [ev[:n4], od[:n4]]),
            "4pcf6": (lambda: lib.gs_count_4pcf6(g._h, p(ev), p(od), 0, len(xyz), st), [ev[:n6], od[:n6]]),
            "4pcf6_weighted": (lambda: lib.gs_count_4pcf6_weighted(g._h, p(ev), p(od), 0, len(xyz), st), [ev, od]),
        }
        sites = {k: _sweep(c, o, torch, monkeypatch) for k, (c, o) in calls.items()}
        assert sites["3pcf_weighted"] >= 1 and sites["4pcf_parity"] >= 1 and sites["4pcf6"] >= 1
        if not windowed:
            ids = torch.arange(len(xyz), dtype=torch.int32, device=dev)
            rp = torch.empty(len(xyz) + 1, dtype=torch.int64, device=dev)
            assert _sweep(lambda: lib.gs_graph_export_rows(g._h, p(ids), len(xyz), p(rp), None, None, st),
                          [rp], torch, monkeypatch) >= 1
            assert _sweep(lambda: lib.gs_count_4pcf_parity_hubs(g._h, p(ids), len(xyz), p(ev), p(od), st),
                          [ev[:n4], od[:n4]], torch, monkeypatch) >= 1
        stats = _lib.GraphStats()
        assert _sweep(lambda: lib.gs_graph_stats(g._h, ctypes.byref(stats), st), [], torch, monkeypatch) >= 1


def test_host_buffer_calls_every_allocation(monkeypatch):
    torch, dev = torch_dev()
    lib = _lib.load()
    xyz, box, periodic, edges = _star(deg=600)
    nb = len(edges) - 1
    n3, n4 = nb * (nb + 1) * (nb + 2) // 6, nb * (nb - 1) * (nb - 2) // 6
    h3 = np.zeros(n3, dtype=np.uint64)
    ev = np.zeros(n4, dtype=np.uint64)
    od = np.zeros(n4, dtype=np.int64)
    ptr = lambda a: a.ctypes.data_as(ctypes.c_void_p)      # noqa: E731
    args = (ptr(xyz), len(xyz), box, periodic, int(edges[-1]), ptr(edges), nb)

    for call, outs in ((lambda: lib.gs_3pcf_from_host(*args, ptr(h3), None), [h3]),
                       (lambda: lib.gs_4pcf_parity_from_host(*args, ptr(ev), ptr(od), None), [ev, od])):
        monkeypatch.delenv("GS_FAULT", raising=False)
        assert call() == _lib.GS_OK
        ref = [o.copy() for o in outs]
        for n in range(1, 64):
            for o in outs:
                o.view(np.uint64)[:] = SENTINEL
            before = _free_bytes(torch)
            monkeypatch.setenv("GS_FAULT", f"alloc:{n}")
            status = call()
            monkeypatch.delenv("GS_FAULT")
            after = _free_bytes(torch)
            if status == _lib.GS_OK:
                assert all(np.array_equal(o, r) for o, r in zip(outs, ref))
                assert n > 5
                break
            assert status == _lib.GS_ERR_NOMEM
            assert all((o.view(np.uint64) == SENTINEL).all() for o in outs)
            assert after == before
        else:
            raise AssertionError("the call never succeeded")
