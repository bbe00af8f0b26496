"""The fixed-workspace parity count against the regular one.

gs_count_4pcf_parity_static exists for callers that must not allocate device
memory while they run -- for example a pipeline that cannot afford the
device-wide synchronisation of cudaMalloc / cudaFree, or a service that
reserves all of its memory up front. It takes its scratch space from a 16 MiB
array compiled into the library instead of allocating it. These tests call it
through the C ABI twice in a row on the same graph and require results
identical (bit for bit: the counts are integers) to gs_count_4pcf_parity and
to the oracle's count over the same input, and they check that the calls
allocate nothing (the library's allocation counter does not move).
This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest

import oracle
from cosmology_point_correlation_gb300 import _lib, catalogues
from tests.gpu_util import gpu_graph, torch_dev

pytestmark = pytest.mark.gpu


def _star_catalogue():
    # one hub with 600 neighbours spread through a ball of 0.98 r_max: its
    # workspace does not fit in shared memory, so the fixed workspace is used
    rng = np.random.default_rng(23)
    R = 20000
    v = rng.normal(size=(600, 3))
    v *= (0.98 * R * rng.uniform(0, 1, size=(600, 1)) ** (1 / 3)) / np.linalg.norm(v, axis=1, keepdims=True)
    xyz = (np.vstack([[[0, 0, 0]], np.rint(v)]) + 100000).astype(np.int32)
    return xyz, 500000, 0, [0, 5000, 9000, 12500, 16000, 18000, R]


def _clustered_catalogue():
    box = catalogues.box_lattice(60.0)
    xyz = catalogues.neyman_scott(6000, 60.0, 120, 50.0, 3.0, 8)
    return xyz, box, 1, catalogues.linear_edges_lu(10.0, 8)


def _count(fn, g, torch, dev, m):
    even = torch.full((m,), -7, dtype=torch.int64, device=dev)      # garbage: outputs must be overwritten
    odd = torch.full((m,), 99, dtype=torch.int64, device=dev)
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    status = fn(g._h, ctypes.c_void_p(even.data_ptr()), ctypes.c_void_p(odd.data_ptr()), 0, g.n, st)
    _lib.check(status)
    torch.cuda.synchronize()
    return even.cpu().numpy(), odd.cpu().numpy()


@pytest.mark.parametrize("make", [_star_catalogue, _clustered_catalogue], ids=["large_hub", "clustered"])
def test_static_workspace_matches_allocating_entry_point(make):
    torch, dev = torch_dev()
    lib = _lib.load()
    xyz, box, periodic, edges = make()
    with gpu_graph(xyz, box, periodic, edges) as g:
        m = len(edges) - 1
        m = m * (m - 1) * (m - 2) // 6
        ref_even, ref_odd = _count(lib.gs_count_4pcf_parity, g, torch, dev, m)
        assert ref_even.sum() > 0
        for _ in range(2):                                        # the workspace is reused
            before = lib.gs_alloc_calls()
            even, odd = _count(lib.gs_count_4pcf_parity_static, g, torch, dev, m)
            assert lib.gs_alloc_calls() == before, "the fixed-workspace call allocated memory"
            assert np.array_equal(even, ref_even)
            assert np.array_equal(odd, ref_odd)
    # the oracle over the same points (the counts do not depend on input order)
    o_even, o_odd = oracle.count_4pcf_parity(xyz, box, periodic, edges)
    assert np.array_equal(even.view(np.uint64), o_even)
    assert np.array_equal(odd, o_odd)


def test_static_workspace_refuses_hubs_too_large():
    # 12,000 points within r_max of each other: a hub of degree 11,999 needs a
    # workspace slice larger than the fixed 16 MiB, so the call must refuse
    torch, dev = torch_dev()
    lib = _lib.load()
    rng = np.random.default_rng(5)
    xyz = (rng.uniform(0, 9000, size=(12000, 3)) + 1000).astype(np.int32)
    with gpu_graph(xyz, 100000, 0, [0, 6000, 12000, 20000]) as g:
        assert g.max_degree == 11999
        even = torch.zeros(1, dtype=torch.int64, device=dev)
        odd = torch.zeros(1, dtype=torch.int64, device=dev)
        st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        status = lib.gs_count_4pcf_parity_static(g._h, ctypes.c_void_p(even.data_ptr()),
                                                 ctypes.c_void_p(odd.data_ptr()), 0, g.n, st)
        assert status == _lib.GS_ERR_CAPACITY
        assert b"static workspace" in lib.gs_last_error()
