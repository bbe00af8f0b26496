"""GB300-native graph-based 3pCF and parity-4pCF counting.

A thin Python layer over libgramsci_gb.so (C ABI: include/gramsci_gb.h). It
only marshals arguments: every step of the computation (cell sort, neighbour
graph, triangle and clique enumeration, histograms) runs in the library's
sm_103a CUDA kernels. PyTorch supplies device memory and CUDA streams.

Counting follows the GRAMSCI v2 paper ("Fast Graph-based Higher-Order
Clustering Statistics on the GPU"): the fixed-radius neighbour graph of §II.1,
the triangle (3pCF) enumeration of §II.2 / §III.1, and the parity-decomposed
4pCF of §III.2 (Eq.(3)).

Histograms come back as int64 tensors whose bits are the library's uint64
counts (torch has no general uint64 arithmetic); use ``as_uint64`` to read
them as unsigned NumPy arrays.
"""
from __future__ import annotations

import ctypes

import numpy as np

from . import _lib
from ._lib import GramsciError

__all__ = ["Graph", "GramsciError", "build_graph", "count_3pcf_from_host",
           "count_4pcf_parity_from_host", "config_count_3pcf", "config_count_4pcf",
           "config_index_3pcf", "config_index_4pcf", "as_uint64", "library_path", "kernel_launches",
           "equilateral", "isosceles", "xi_natural", "config_tuples_4pcf6", "zeta4_disconnected",
           "as_int128", "xi_signed", "zeta4_connected", "measure_smem_atomics",
           "quantize_weights", "WEIGHT_SCALE"]


def library_path() -> str:
    return _lib.lib_path()


def kernel_launches() -> int:
    """Kernels the library has launched in this process."""
    return int(_lib.load().gs_kernel_launches())


def measure_smem_atomics(ncfg: int, pattern: int = 0, lanes_active: int = 32, stream=None) -> float:
    """Lane-adds per second the device retires when its SMs do nothing but
    shared-memory atomic adds into a histogram of ncfg 32-bit counters
    (pattern 0: random counters, 1: one bank per lane, 2: one counter)."""
    v = ctypes.c_double()
    _lib.check(_lib.load().gs_measure_smem_atomics(int(ncfg), int(pattern), int(lanes_active),
                                                   ctypes.byref(v), _stream(stream)))
    return v.value


def _torch():
    import torch
    return torch


def _stream(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _edges(edges_lu):
    e = np.ascontiguousarray(np.asarray(edges_lu, dtype=np.int64))
    if e.ndim != 1 or len(e) < 2:
        raise ValueError("edges_lu needs at least two entries")
    return e


def as_uint64(t) -> np.ndarray:
    """Host NumPy uint64 view of a histogram tensor."""
    return t.detach().cpu().numpy().view(np.uint64)


WEIGHT_SCALE = 32767


def quantize_weights(w) -> np.ndarray:
    """int16 fixed-point weights for set_weights from real weights |w| <= 1:
    q = round(WEIGHT_SCALE w). Each weight moves by at most 1/(2 WEIGHT_SCALE),
    so a product of k weights (a pair, triangle or tetrahedron term) moves by
    at most k/(2 WEIGHT_SCALE), and a weighted sum over n terms, divided by
    WEIGHT_SCALE^k, is within n k/(2 WEIGHT_SCALE) of the sum of the real
    weights' products. Weights of larger modulus must be rescaled first."""
    w = np.asarray(w, dtype=np.float64)
    if not np.all(np.isfinite(w)) or np.any(np.abs(w) > 1.0):
        raise ValueError("weights must be finite with |w| <= 1 (rescale them first)")
    return np.rint(w * WEIGHT_SCALE).astype(np.int16)


def as_int128(t) -> list:
    """Python ints from 128-bit two's-complement (low, high) int64 word pairs
    (the weighted counts' output, shape [m, 2])."""
    w = np.asarray(t.cpu().numpy() if hasattr(t, "cpu") else t, dtype=np.int64).reshape(-1, 2)
    return [(int(hi) << 64) + (int(lo) & 0xFFFFFFFFFFFFFFFF) for lo, hi in w]


def config_count_3pcf(nbins: int) -> int:
    return _lib.load().gs_config_count_3pcf(nbins)


def config_count_4pcf(nbins: int) -> int:
    return _lib.load().gs_config_count_4pcf(nbins)


def config_index_3pcf(nbins: int, b1: int, b2: int, b3: int) -> int:
    return _lib.load().gs_config_index_3pcf(nbins, b1, b2, b3)


def config_index_4pcf(nbins: int, b1: int, b2: int, b3: int) -> int:
    return _lib.load().gs_config_index_4pcf(nbins, b1, b2, b3)


class Graph:
    """A neighbour graph resident in device memory (handle of the C library)."""

    def __init__(self, handle: ctypes.c_void_p, nbins: int, device):
        self._h = handle
        self.nbins = nbins
        self.device = device

    # -- sizes
    def info(self):
        n, e, m = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32()
        _lib.check(_lib.load().gs_graph_info(self._h, ctypes.byref(n), ctypes.byref(e), ctypes.byref(m)))
        return n.value, e.value, m.value

    @property
    def n(self) -> int:
        return self.info()[0]

    @property
    def n_edges(self) -> int:
        return self.info()[1]

    @property
    def max_degree(self) -> int:
        return self.info()[2]

    def windows(self):
        """(number of row windows, largest window's edges); 0 windows = device-resident."""
        nw, m = ctypes.c_int32(), ctypes.c_int64()
        _lib.check(_lib.load().gs_graph_windows(self._h, ctypes.byref(nw), ctypes.byref(m)))
        return nw.value, m.value

    def stats(self, stream=None) -> dict:
        """Work statistics (sum C(f,2), sum b*f, max forward degree, ...); synchronises."""
        st = _lib.GraphStats()
        _lib.check(_lib.load().gs_graph_stats(self._h, ctypes.byref(st), _stream(stream)))
        return {name: getattr(st, name) for name, _ in _lib.GraphStats._fields_ if name != "reserved"}

    def hub_work(self, stream=None):
        """(f int32 [n], w int64 [n]) per hub in internal order: the forward degree
        and the spoke-row entries of the hub's 3pCF merge-walks (sum of f_j over
        its forward spokes j)."""
        torch = _torch()
        n = self.n
        f = torch.empty(max(n, 1), dtype=torch.int32, device=self.device)
        w = torch.empty(max(n, 1), dtype=torch.int64, device=self.device)
        _lib.check(_lib.load().gs_graph_hub_work(self._h, ctypes.c_void_p(f.data_ptr()),
                                                 ctypes.c_void_p(w.data_ptr()), _stream(stream)))
        return f[:n], w[:n]

    # -- counts
    def count_2pcf(self, out=None, stream=None):
        """Unordered pairs per radial bin (uint64 bits in an int64 tensor)."""
        torch = _torch()
        if out is None:
            out = torch.empty(self.nbins, dtype=torch.int64, device=self.device)
        _lib.check(_lib.load().gs_count_2pcf(self._h, ctypes.c_void_p(out.data_ptr()), _stream(stream)))
        return out

    def set_weights(self, weights, stream=None):
        """Attach int16 fixed-point point weights (input order, a CUDA tensor [n])
        for the weighted counts; the library keeps its own copy."""
        torch = _torch()
        if not (isinstance(weights, torch.Tensor) and weights.is_cuda and weights.dtype == torch.int16):
            raise TypeError("weights must be an int16 CUDA tensor of shape [n]")
        weights = weights.contiguous().reshape(-1)
        if weights.numel() != self.n:
            raise ValueError(f"weights has {weights.numel()} entries, the graph {self.n} points")
        _lib.check(_lib.load().gs_graph_set_weights(self._h, ctypes.c_void_p(weights.data_ptr()), _stream(stream)))

    def count_2pcf_weighted(self, out=None, stream=None):
        """Per bin, the exact sum of w_i w_j over pairs: int64 tensor [nbins, 2] of
        (low, high) words of a 128-bit integer (see as_int128)."""
        torch = _torch()
        if out is None:
            out = torch.empty((self.nbins, 2), dtype=torch.int64, device=self.device)
        _lib.check(_lib.load().gs_count_2pcf_weighted(self._h, ctypes.c_void_p(out.data_ptr()), _stream(stream)))
        return out

    def count_3pcf_weighted(self, hub_begin: int = 0, hub_end: int | None = None, out=None, stream=None):
        """Per sorted-bin configuration, the exact sum of w_i w_j w_k over triangles:
        int64 tensor [n_configs, 2] of 128-bit (low, high) words (see as_int128)."""
        torch = _torch()
        hub_end = self.n if hub_end is None else hub_end
        if out is None:
            out = torch.empty((config_count_3pcf(self.nbins), 2), dtype=torch.int64, device=self.device)
        _lib.check(_lib.load().gs_count_3pcf_weighted(self._h, ctypes.c_void_p(out.data_ptr()),
                                                      int(hub_begin), int(hub_end), _stream(stream)))
        return out

    def count_4pcf6_weighted(self, hub_begin: int = 0, hub_end: int | None = None, stream=None):
        """Weighted six-bin 4pCF: (even, odd) int64 tensors [n_configs, 2] of
        128-bit (low, high) words: sums of w_i w_j w_k w_l and of the odd sign
        times that product (see as_int128)."""
        torch = _torch()
        if self.nbins > 10:
            raise GramsciError(_lib.GS_ERR_ARG, "the six-bin 4pCF supports at most 10 bins")
        hub_end = self.n if hub_end is None else hub_end
        m = _lib.load().gs_config_count_4pcf6(self.nbins)
        even = torch.empty((m, 2), dtype=torch.int64, device=self.device)
        odd = torch.empty((m, 2), dtype=torch.int64, device=self.device)
        _lib.check(_lib.load().gs_count_4pcf6_weighted(self._h, ctypes.c_void_p(even.data_ptr()),
                                                       ctypes.c_void_p(odd.data_ptr()), int(hub_begin),
                                                       int(hub_end), _stream(stream)))
        return even, odd

    @property
    def count3_walk(self) -> str:
        """The spoke walk count_3pcf takes on this graph: "map", "mapgroup", "group" or "warp"."""
        return {3: "mapgroup", 2: "map", 1: "group", 0: "warp"}.get(_lib.load().gs_count3_walk(self._h), "?")

    def count_3pcf(self, hub_begin: int = 0, hub_end: int | None = None, out=None, stream=None):
        """uint64 triangle histogram over sorted bin triples (int64 tensor on the device).

        The library picks the spoke walk from the graph (count3_walk); the
        environment variable GS_COUNT3_WALK = "map", "mapgroup", "group" or
        "warp" fixes it. Results are identical."""
        torch = _torch()
        hub_end = self.n if hub_end is None else hub_end
        m = config_count_3pcf(self.nbins)
        if out is None:
            out = torch.empty(m, dtype=torch.int64, device=self.device)
        _lib.check(_lib.load().gs_count_3pcf(self._h, ctypes.c_void_p(out.data_ptr()),
                                             int(hub_begin), int(hub_end), _stream(stream)))
        return out

    def count_4pcf_parity(self, hub_begin: int = 0, hub_end: int | None = None, out=None, stream=None):
        """(even uint64, odd int64) histograms over strictly increasing hub-bin triples."""
        torch = _torch()
        hub_end = self.n if hub_end is None else hub_end
        m = max(config_count_4pcf(self.nbins), 0)
        if out is None:
            out = (torch.zeros(m, dtype=torch.int64, device=self.device),
                   torch.zeros(m, dtype=torch.int64, device=self.device))
        even, odd = out
        _lib.check(_lib.load().gs_count_4pcf_parity(self._h, ctypes.c_void_p(even.data_ptr()),
                                                    ctypes.c_void_p(odd.data_ptr()),
                                                    int(hub_begin), int(hub_end), _stream(stream)))
        return even, odd

    def count_4pcf6(self, hub_begin: int = 0, hub_end: int | None = None, out=None, stream=None):
        """(even, odd) six-edge-bin 4pCF per tetrahedron configuration (each tetrahedron once)."""
        torch = _torch()
        hub_end = self.n if hub_end is None else hub_end
        m = _lib.load().gs_config_count_4pcf6(self.nbins)
        if m < 0:
            raise GramsciError(_lib.GS_ERR_ARG, "the six-bin 4pCF supports at most 10 bins")
        if out is None:
            out = (torch.zeros(m, dtype=torch.int64, device=self.device),
                   torch.zeros(m, dtype=torch.int64, device=self.device))
        even, odd = out
        _lib.check(_lib.load().gs_count_4pcf6(self._h, ctypes.c_void_p(even.data_ptr()),
                                              ctypes.c_void_p(odd.data_ptr()), int(hub_begin), int(hub_end),
                                              _stream(stream)))
        return even, odd

    def count_3pcf_hubs(self, hubs, out=None, stream=None):
        """Triangles incident to each listed hub (input indices), summed; uint64 bits in int64."""
        torch = _torch()
        h = _ids(hubs, self.device)
        m = config_count_3pcf(self.nbins)
        if out is None:
            out = torch.empty(m, dtype=torch.int64, device=self.device)
        _lib.check(_lib.load().gs_count_3pcf_hubs(self._h, ctypes.c_void_p(h.data_ptr()), h.numel(),
                                                  ctypes.c_void_p(out.data_ptr()), _stream(stream)))
        return out

    def count_4pcf_parity_hubs(self, hubs, out=None, stream=None):
        """(even, odd) parity-4pCF contribution of the listed hubs (input indices)."""
        torch = _torch()
        h = _ids(hubs, self.device)
        m = max(config_count_4pcf(self.nbins), 0)
        if out is None:
            out = (torch.zeros(m, dtype=torch.int64, device=self.device),
                   torch.zeros(m, dtype=torch.int64, device=self.device))
        even, odd = out
        _lib.check(_lib.load().gs_count_4pcf_parity_hubs(self._h, ctypes.c_void_p(h.data_ptr()), h.numel(),
                                                         ctypes.c_void_p(even.data_ptr()),
                                                         ctypes.c_void_p(odd.data_ptr()), _stream(stream)))
        return even, odd

    def export_rows(self, ids, stream=None):
        """(row_ptr int64 [count+1], nbr int32, bin uint8) of the listed input points, sorted rows."""
        torch = _torch()
        h = _ids(ids, self.device)
        row_ptr = torch.empty(h.numel() + 1, dtype=torch.int64, device=self.device)
        lib = _lib.load()
        _lib.check(lib.gs_graph_export_rows(self._h, ctypes.c_void_p(h.data_ptr()), h.numel(),
                                            ctypes.c_void_p(row_ptr.data_ptr()), None, None, _stream(stream)))
        total = int(row_ptr[-1].item())
        nbr = torch.empty(max(total, 1), dtype=torch.int32, device=self.device)
        bins = torch.empty(max(total, 1), dtype=torch.uint8, device=self.device)
        _lib.check(lib.gs_graph_export_rows(self._h, ctypes.c_void_p(h.data_ptr()), h.numel(),
                                            ctypes.c_void_p(row_ptr.data_ptr()), ctypes.c_void_p(nbr.data_ptr()),
                                            ctypes.c_void_p(bins.data_ptr()), _stream(stream)))
        return row_ptr, nbr[:total], bins[:total]

    # -- exports
    def export_csr(self, stream=None):
        """(row_ptr int64 [n+1], nbr int32 [E], bin uint8 [E]) in input numbering, rows sorted."""
        torch = _torch()
        n, e, _ = self.info()
        row_ptr = torch.empty(n + 1, dtype=torch.int64, device=self.device)
        nbr = torch.empty(max(e, 1), dtype=torch.int32, device=self.device)
        bins = torch.empty(max(e, 1), dtype=torch.uint8, device=self.device)
        _lib.check(_lib.load().gs_graph_export_csr(self._h, ctypes.c_void_p(row_ptr.data_ptr()),
                                                   ctypes.c_void_p(nbr.data_ptr()),
                                                   ctypes.c_void_p(bins.data_ptr()), _stream(stream)))
        return row_ptr, nbr[:e], bins[:e]

    def export_perm(self, stream=None):
        """int32 [n]: input index of each point in the graph's internal (hub) order."""
        torch = _torch()
        perm = torch.empty(max(self.n, 1), dtype=torch.int32, device=self.device)
        _lib.check(_lib.load().gs_graph_export_perm(self._h, ctypes.c_void_p(perm.data_ptr()),
                                                    _stream(stream)))
        return perm[:self.n]

    def free(self):
        if self._h:
            _lib.load().gs_graph_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.free()


def equilateral(hist, nbins: int):
    """The equilateral slice of a 3pCF histogram: configurations (b, b, b), b = 0..nbins-1."""
    h = np.asarray(hist)
    return h[[config_index_3pcf(nbins, b, b, b) for b in range(nbins)]]


def isosceles(hist, nbins: int, b: int):
    """Configurations with two sides in bin b: entry c is the sorted triple of (b, b, c)."""
    h = np.asarray(hist)
    return h[[config_index_3pcf(nbins, *sorted((b, b, c))) for c in range(nbins)]]


def xi_natural(dd, rr, n_data: int, n_random: int):
    """Natural-estimator 2pCF per bin from data and random pair counts:
    xi = (DD / C(n_data, 2)) / (RR / C(n_random, 2)) - 1."""
    dd = np.asarray(dd, dtype=np.float64)
    rr = np.asarray(rr, dtype=np.float64)
    nd = n_data * (n_data - 1) / 2.0
    nr = n_random * (n_random - 1) / 2.0
    with np.errstate(divide="ignore", invalid="ignore"):
        return (dd / nd) / (rr / nr) - 1.0


def config_tuples_4pcf6(nbins: int) -> np.ndarray:
    """int32 [n_configs, 6]: the smallest bin tuple (b01, b02, b03, b12, b13, b23)
    of every six-bin 4pCF configuration, in index order."""
    lib = _lib.load()
    n = lib.gs_config_count_4pcf6(nbins)
    if n < 0:
        raise GramsciError(_lib.GS_ERR_ARG, "nbins outside 1..10")
    out = np.zeros((n, 6), dtype=np.int32)
    for c in range(n):
        _lib.check(lib.gs_config_tuple_4pcf6(nbins, c, out[c].ctypes.data_as(ctypes.c_void_p)))
    return out


def zeta4_disconnected(xi, nbins: int) -> np.ndarray:
    """Disconnected 4pCF of every six-bin configuration (GRAMSCI v2 §III.3,
    Eq.(4)): xi(r01) xi(r23) + xi(r02) xi(r13) + xi(r03) xi(r12), the sum over
    the three ways of splitting the four points into two pairs, evaluated on
    the configuration's bins; xi is the binned 2pCF (length nbins)."""
    x = np.asarray(xi, dtype=np.float64)
    t = config_tuples_4pcf6(nbins)
    return x[t[:, 0]] * x[t[:, 5]] + x[t[:, 1]] * x[t[:, 4]] + x[t[:, 2]] * x[t[:, 3]]


def xi_signed(pair_sums, rr):
    """2pCF per bin from the signed-weight pair sums (GRAMSCI v2 §III.3): with
    data weights summing to +1 and random weights to -1 the pair sum is the
    Landy-Szalay numerator DD - 2DR + RR, so xi = (signed pair sum) / RR. Both
    arguments are per-bin sums in the same weight units (e.g. as_int128 of
    count_2pcf_weighted on the joint catalogue, and on the randoms alone)."""
    s = np.array([float(v) for v in pair_sums], dtype=np.float64)
    r = np.array([float(v) for v in rr], dtype=np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        return s / r


def zeta4_connected(nnnn, rrrr, xi, nbins: int) -> np.ndarray:
    """Connected six-bin 4pCF, Eq.(5): zeta = NNNN / RRRR per configuration
    minus the disconnected part of Eq.(4) built from the binned xi. NNNN is the
    even channel of count_4pcf6_weighted on the joint catalogue, RRRR the same
    count on the randoms alone (same weight units). The odd channel needs no
    subtraction: NNNN_odd / RRRR is already connected."""
    n = np.array([float(v) for v in nnnn], dtype=np.float64)
    r = np.array([float(v) for v in rrrr], dtype=np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        zeta = n / r
    return zeta - zeta4_disconnected(xi, nbins)


def _ids(ids, device):
    torch = _torch()
    t = torch.as_tensor(np.asarray(ids, dtype=np.int32) if not isinstance(ids, torch.Tensor) else ids)
    return t.to(device=device, dtype=torch.int32).contiguous().reshape(-1)


def build_graph(coords, box_lu: int, periodic: bool, edges_lu, stream=None,
                window_edges: int | None = None) -> Graph:
    """Neighbour graph of int32 lattice coordinates (a CUDA tensor [n, 3]).
    window_edges: keep the edge arrays in pinned host memory, in row windows of
    at most this many directed edges (out-of-core mode)."""
    torch = _torch()
    if not (isinstance(coords, torch.Tensor) and coords.is_cuda and coords.dtype == torch.int32):
        raise TypeError("coords must be an int32 CUDA tensor of shape [n, 3]")
    coords = coords.contiguous().reshape(-1, 3)
    e = _edges(edges_lu)
    h = ctypes.c_void_p()
    lib = _lib.load()
    args = (ctypes.c_void_p(coords.data_ptr()), coords.shape[0], int(box_lu), int(bool(periodic)), int(e[-1]),
            e.ctypes.data_as(ctypes.c_void_p), len(e) - 1)
    if window_edges is None:
        _lib.check(lib.gs_build_graph(*args, _stream(stream), ctypes.byref(h)))
    else:
        _lib.check(lib.gs_build_graph_windowed(*args, int(window_edges), _stream(stream), ctypes.byref(h)))
    return Graph(h, len(e) - 1, coords.device)


def count_3pcf_from_host(coords: np.ndarray, box_lu: int, periodic: bool, edges_lu, out=None,
                         stream=None) -> np.ndarray:
    """Host coordinates in, host uint64 histogram out, in one library call."""
    xyz = np.ascontiguousarray(np.asarray(coords, dtype=np.int32).reshape(-1, 3))
    e = _edges(edges_lu)
    m = config_count_3pcf(len(e) - 1)
    if out is None:
        out = np.zeros(m, dtype=np.uint64)
    _lib.check(_lib.load().gs_3pcf_from_host(xyz.ctypes.data_as(ctypes.c_void_p), len(xyz), int(box_lu),
                                             int(bool(periodic)), int(e[-1]), e.ctypes.data_as(ctypes.c_void_p),
                                             len(e) - 1, out.ctypes.data_as(ctypes.c_void_p), _stream(stream)))
    return out


def count_4pcf_parity_from_host(coords: np.ndarray, box_lu: int, periodic: bool, edges_lu, out=None,
                                stream=None):
    xyz = np.ascontiguousarray(np.asarray(coords, dtype=np.int32).reshape(-1, 3))
    e = _edges(edges_lu)
    m = max(config_count_4pcf(len(e) - 1), 0)
    if out is None:
        out = (np.zeros(max(m, 1), dtype=np.uint64), np.zeros(max(m, 1), dtype=np.int64))
    even, odd = out
    _lib.check(_lib.load().gs_4pcf_parity_from_host(
        xyz.ctypes.data_as(ctypes.c_void_p), len(xyz), int(box_lu), int(bool(periodic)), int(e[-1]),
        e.ctypes.data_as(ctypes.c_void_p), len(e) - 1, even.ctypes.data_as(ctypes.c_void_p),
        odd.ctypes.data_as(ctypes.c_void_p), _stream(stream)))
    return even[:m], odd[:m]
