"""Helpers for the GPU tests: run the library on NumPy inputs, return NumPy."""
import numpy as np

import oracle


def torch_dev():
    import torch
    return torch, torch.device("cuda:0")


def gpu_graph(xyz, box, periodic, edges):
    from cosmology_point_correlation_gb300 import build_graph
    torch, dev = torch_dev()
    return build_graph(torch.from_numpy(np.ascontiguousarray(xyz, dtype=np.int32)).to(dev),
                       box, periodic, edges)


def gpu_csr(xyz, box, periodic, edges):
    with gpu_graph(xyz, box, periodic, edges) as g:
        rp, nbr, b = g.export_csr()
        info = g.info()
        return rp.cpu().numpy(), nbr.cpu().numpy(), b.cpu().numpy(), info


def gpu_3pcf(xyz, box, periodic, edges, ranges=None):
    from cosmology_point_correlation_gb300 import as_uint64
    with gpu_graph(xyz, box, periodic, edges) as g:
        if ranges is None:
            return as_uint64(g.count_3pcf())
        return [as_uint64(g.count_3pcf(a, b)) for a, b in ranges]


def gpu_4pcf(xyz, box, periodic, edges, ranges=None):
    from cosmology_point_correlation_gb300 import as_uint64
    with gpu_graph(xyz, box, periodic, edges) as g:
        if ranges is None:
            e, o = g.count_4pcf_parity()
            return as_uint64(e), o.cpu().numpy()
        out = []
        for a, b in ranges:
            e, o = g.count_4pcf_parity(a, b)
            out.append((as_uint64(e), o.cpu().numpy()))
        return out


def assert_graph_equal(xyz, box, periodic, edges):
    rp, nbr, b, (n, e, maxd) = gpu_csr(xyz, box, periodic, edges)
    ref = oracle.graph(xyz, box, periodic, edges)
    assert n == len(xyz)
    assert e == ref.n_edges
    assert np.array_equal(rp, ref.row_ptr)
    assert np.array_equal(nbr, ref.nbr)
    assert np.array_equal(b, ref.bin)
    deg = np.diff(ref.row_ptr)
    assert maxd == (int(deg.max()) if len(deg) else 0)
    return ref


def mirror(xyz, box, periodic):
    m = xyz.astype(np.int64).copy()
    m[:, 0] = (box - m[:, 0]) % box if periodic else box - 1 - m[:, 0]
    return m.astype(np.int32)
