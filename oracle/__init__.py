"""CPU oracle for graph-based 3pCF and parity-4pCF counts (ctypes over gs_oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline use it; the library's product path never imports it. It shares no
code with the CUDA library. Every function follows the GRAMSCI v2 paper
("Fast Graph-based Higher-Order Clustering Statistics on the GPU"):

- ``graph``: brute-force neighbour lists, sorted (§II.1, Eq.(1)), with bin bytes.
- ``count_3pcf``: hub-and-spoke triangle loop (§II.2), one count per unordered
  triangle, sorted bin triple packed lexicographically (§V.1, Fig.8 key).
- ``count_4pcf_parity``: even count and odd sum of sign(V), V from Eq.(3),
  with V == 0 giving odd weight 0 (§III.2).
- ``brute3`` / ``brute4``: all triples / quadruples with no graph.
- ``count_4pcf6`` / ``brute4six``: six-edge-bin 4pCF (each tetrahedron once, its
  configuration the smallest bin tuple over vertex orderings, odd channel the
  sign of V for a minimal ordering of a chiral configuration; §II.2, §III.2,
  276 configurations for 4 bins as in §V.2).
- ``count_2pcf_weighted`` / ``count_3pcf_weighted``: exact sums of products of
  signed integer weights (§II.1, §III.3: the Landy-Szalay / Szapudi-Szalay
  numerators), in 128-bit integers.
- ``row``, ``count_3pcf_hubs``, ``count_4pcf_parity_hubs``: per point / per hub
  results from brute-force rows, for sampled checks at full size.

Parity pins: every function here is checked in ``tests/test_oracle_*.py``
against hand-derived fixtures, closed forms, invariants and an independent
NumPy brute force; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# GS_ORACLE_SRC / GS_ORACLE_LIB point the wrapper at another copy of the C
# source and library. Only tests/test_oracle_mutants.py sets them, to run the
# pins against copies with a planted mistake.
_SRC = os.environ.get("GS_ORACLE_SRC") or os.path.join(_HERE, "gs_oracle.c")
_LIB = os.environ.get("GS_ORACLE_LIB") or os.path.join(_HERE, "liboracle.so")
_lib = None

_i64 = ctypes.c_int64
_int = ctypes.c_int
_p = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile gs_oracle.c into oracle/liboracle.so (plain gcc, pthreads)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-Wall", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        cat = [_p, _i64, _i64, _int, _p, _int]
        lib.oracle_graph_degrees.argtypes = cat + [_p]
        lib.oracle_graph_degrees.restype = _i64
        lib.oracle_graph_fill.argtypes = cat + [_p, _p, _p]
        lib.oracle_row.argtypes = cat + [_i64, _p, _p]
        lib.oracle_row.restype = _i64
        lib.oracle_3pcf_range.argtypes = cat + [_p, _p, _p, _i64, _i64, _p]
        lib.oracle_4pcf_parity_range.argtypes = cat + [_p, _p, _p, _i64, _i64, _p, _p]
        lib.oracle_4pcf_parity_hubs.argtypes = cat + [_p, _i64, _p, _p]
        lib.oracle_3pcf_hubs.argtypes = cat + [_p, _i64, _p]
        lib.oracle_4pcf6.argtypes = cat + [_p, _p, _i64, _i64, _p, _p]
        lib.oracle_2pcf_weighted.argtypes = cat + [_p, _p]
        lib.oracle_3pcf_weighted.argtypes = cat + [_p, _p, _p, _p, _p]
        lib.oracle_4pcf6_weighted.argtypes = cat + [_p, _p, _p, _i64, _i64, _p, _p]
        lib.oracle_brute4six.argtypes = cat + [_p, _p]
        lib.oracle_nconfig6.argtypes = [_int]
        lib.oracle_nconfig6.restype = _i64
        lib.oracle_config_index6.argtypes = [_int, _p]
        lib.oracle_config_index6.restype = _i64
        lib.oracle_brute3.argtypes = cat + [_p]
        lib.oracle_brute4.argtypes = cat + [_p, _p]
        lib.oracle_nconfig3.argtypes = [_int]
        lib.oracle_nconfig3.restype = _i64
        lib.oracle_nconfig4.argtypes = [_int]
        lib.oracle_nconfig4.restype = _i64
        lib.oracle_threads.restype = _int
        lib.oracle_set_threads.argtypes = [_int]
        lib.oracle_set_threads.restype = _int
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _cat(xyz, box_lu, periodic, edges_lu):
    xyz = np.ascontiguousarray(np.asarray(xyz, dtype=np.int32).reshape(-1, 3))
    edges = np.ascontiguousarray(np.asarray(edges_lu, dtype=np.int64))
    nb = len(edges) - 1
    if nb < 1:
        raise ValueError("need at least one bin")
    return xyz, edges, nb, [_ptr(xyz), len(xyz), int(box_lu), int(bool(periodic)), _ptr(edges), nb]


def threads() -> int:
    return _load().oracle_threads()


def set_threads(t: int) -> int:
    return _load().oracle_set_threads(int(t))


def nconfig3(nb: int) -> int:
    return _load().oracle_nconfig3(nb)


def nconfig4(nb: int) -> int:
    return _load().oracle_nconfig4(nb)


class Graph:
    """Brute-force CSR graph in input numbering."""

    def __init__(self, row_ptr, nbr, bin_):
        self.row_ptr, self.nbr, self.bin = row_ptr, nbr, bin_

    @property
    def n_edges(self) -> int:
        return int(self.row_ptr[-1])


def graph(xyz, box_lu, periodic, edges_lu) -> Graph:
    lib = _load()
    xyz, edges, nb, cat = _cat(xyz, box_lu, periodic, edges_lu)
    n = len(xyz)
    deg = np.zeros(n, dtype=np.int64)
    e = lib.oracle_graph_degrees(*cat, _ptr(deg))
    row_ptr = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(deg, out=row_ptr[1:])
    assert row_ptr[-1] == e
    nbr = np.zeros(max(e, 1), dtype=np.int32)
    bin_ = np.zeros(max(e, 1), dtype=np.uint8)
    lib.oracle_graph_fill(*cat, _ptr(row_ptr), _ptr(nbr), _ptr(bin_))
    return Graph(row_ptr, nbr[:e], bin_[:e])


def row(xyz, box_lu, periodic, edges_lu, i: int):
    """N(i) and its bins, by brute force over all points."""
    lib = _load()
    xyz, edges, nb, cat = _cat(xyz, box_lu, periodic, edges_lu)
    nbr = np.zeros(max(len(xyz), 1), dtype=np.int32)
    bin_ = np.zeros(max(len(xyz), 1), dtype=np.uint8)
    m = lib.oracle_row(*cat, int(i), _ptr(nbr), _ptr(bin_))
    return nbr[:m].copy(), bin_[:m].copy()


def _graph_args(g: Graph):
    nbr = g.nbr if len(g.nbr) else np.zeros(1, dtype=np.int32)
    bin_ = g.bin if len(g.bin) else np.zeros(1, dtype=np.uint8)
    return [_ptr(g.row_ptr), _ptr(nbr), _ptr(bin_)], (nbr, bin_)


def count_3pcf(xyz, box_lu, periodic, edges_lu, g: Graph | None = None,
               hub_begin: int = 0, hub_end: int | None = None) -> np.ndarray:
    lib = _load()
    xyz, edges, nb, cat = _cat(xyz, box_lu, periodic, edges_lu)
    if g is None:
        g = graph(xyz, box_lu, periodic, edges)
    hub_end = len(xyz) if hub_end is None else hub_end
    hist = np.zeros(nconfig3(nb), dtype=np.uint64)
    gargs, keep = _graph_args(g)
    lib.oracle_3pcf_range(*cat, *gargs, int(hub_begin), int(hub_end), _ptr(hist))
    return hist


def count_4pcf_parity(xyz, box_lu, periodic, edges_lu, g: Graph | None = None,
                      hub_begin: int = 0, hub_end: int | None = None):
    lib = _load()
    xyz, edges, nb, cat = _cat(xyz, box_lu, periodic, edges_lu)
    if g is None:
        g = graph(xyz, box_lu, periodic, edges)
    hub_end = len(xyz) if hub_end is None else hub_end
    m = max(nconfig4(nb), 0)
    even = np.zeros(max(m, 1), dtype=np.uint64)
    odd = np.zeros(max(m, 1), dtype=np.int64)
    gargs, keep = _graph_args(g)
    lib.oracle_4pcf_parity_range(*cat, *gargs, int(hub_begin), int(hub_end),
                                 _ptr(even), _ptr(odd))
    return even[:m], odd[:m]


def count_2pcf(xyz, box_lu, periodic, edges_lu, g: Graph | None = None) -> np.ndarray:
    """Unordered pairs per radial bin: each pair sits in two rows of the graph."""
    xyz, edges, nb, _ = _cat(xyz, box_lu, periodic, edges_lu)
    if g is None:
        g = graph(xyz, box_lu, periodic, edges)
    return (np.bincount(g.bin, minlength=nb) // 2).astype(np.uint64)


def nconfig6(nb: int) -> int:
    """Six-edge-bin tetrahedron configurations for nb bins (by enumeration)."""
    return _load().oracle_nconfig6(nb)


def config_index6(nb: int, t) -> int:
    """Index of a canonical tuple (b01, b02, b03, b12, b13, b23); -1 if not canonical."""
    a = np.ascontiguousarray(np.asarray(t, dtype=np.int32))
    return _load().oracle_config_index6(nb, _ptr(a))


def count_4pcf6(xyz, box_lu, periodic, edges_lu, g: Graph | None = None,
                hub_begin: int = 0, hub_end: int | None = None):
    """Six-edge-bin 4pCF: (even, odd) per configuration, each tetrahedron once
    (at its lowest-index vertex; hub range in input numbering)."""
    lib = _load()
    xyz, edges, nb, cat = _cat(xyz, box_lu, periodic, edges_lu)
    if g is None:
        g = graph(xyz, box_lu, periodic, edges)
    hub_end = len(xyz) if hub_end is None else hub_end
    m = nconfig6(nb)
    even = np.zeros(m, dtype=np.uint64)
    odd = np.zeros(m, dtype=np.int64)
    nbr = g.nbr if len(g.nbr) else np.zeros(1, dtype=np.int32)
    lib.oracle_4pcf6(*cat, _ptr(g.row_ptr), _ptr(nbr), int(hub_begin), int(hub_end), _ptr(even), _ptr(odd))
    return even, odd


def brute4six(xyz, box_lu, periodic, edges_lu):
    lib = _load()
    xyz, edges, nb, cat = _cat(xyz, box_lu, periodic, edges_lu)
    m = nconfig6(nb)
    even = np.zeros(m, dtype=np.uint64)
    odd = np.zeros(m, dtype=np.int64)
    lib.oracle_brute4six(*cat, _ptr(even), _ptr(odd))
    return even, odd


def from_words128(words) -> list:
    """Python ints from (low, high) int64 word pairs."""
    a = np.asarray(words, dtype=np.int64).reshape(-1, 2)
    return [int(lo) % (1 << 64) + (int(hi) << 64) for lo, hi in a]


def count_2pcf_weighted(xyz, box_lu, periodic, edges_lu, w) -> list:
    """Exact sum of w_i w_j over the pairs of each bin (Python ints); brute force."""
    lib = _load()
    xyz, edges, nb, cat = _cat(xyz, box_lu, periodic, edges_lu)
    w = np.ascontiguousarray(np.asarray(w, dtype=np.int16))
    out = np.zeros(2 * nb, dtype=np.int64)
    lib.oracle_2pcf_weighted(*cat, _ptr(w), _ptr(out))
    return from_words128(out)


def count_3pcf_weighted(xyz, box_lu, periodic, edges_lu, w, g: Graph | None = None) -> list:
    """Exact sum of w_i w_j w_k over the triangles of each configuration (Python ints)."""
    lib = _load()
    xyz, edges, nb, cat = _cat(xyz, box_lu, periodic, edges_lu)
    if g is None:
        g = graph(xyz, box_lu, periodic, edges)
    w = np.ascontiguousarray(np.asarray(w, dtype=np.int16))
    out = np.zeros(2 * nconfig3(nb), dtype=np.int64)
    gargs, keep = _graph_args(g)
    lib.oracle_3pcf_weighted(*cat, *gargs, _ptr(w), _ptr(out))
    return from_words128(out)


def count_4pcf6_weighted(xyz, box_lu, periodic, edges_lu, w, g: Graph | None = None,
                         hub_begin: int = 0, hub_end: int | None = None):
    """Weighted six-bin 4pCF: (even, odd) lists of Python ints per configuration,
    the exact sums of w_i w_j w_k w_l and of sign x w_i w_j w_k w_l."""
    lib = _load()
    xyz, edges, nb, cat = _cat(xyz, box_lu, periodic, edges_lu)
    if g is None:
        g = graph(xyz, box_lu, periodic, edges)
    hub_end = len(xyz) if hub_end is None else hub_end
    w = np.ascontiguousarray(np.asarray(w, dtype=np.int16))
    m = nconfig6(nb)
    even = np.zeros(2 * m, dtype=np.int64)
    odd = np.zeros(2 * m, dtype=np.int64)
    nbr = g.nbr if len(g.nbr) else np.zeros(1, dtype=np.int32)
    lib.oracle_4pcf6_weighted(*cat, _ptr(g.row_ptr), _ptr(nbr), _ptr(w), int(hub_begin), int(hub_end),
                              _ptr(even), _ptr(odd))
    return from_words128(even), from_words128(odd)


def count_3pcf_hubs(xyz, box_lu, periodic, edges_lu, hubs) -> np.ndarray:
    """Triangles incident to each listed hub (input numbering), summed; no graph."""
    lib = _load()
    xyz, edges, nb, cat = _cat(xyz, box_lu, periodic, edges_lu)
    hubs = np.ascontiguousarray(np.asarray(hubs, dtype=np.int64))
    hist = np.zeros(nconfig3(nb), dtype=np.uint64)
    lib.oracle_3pcf_hubs(*cat, _ptr(hubs), len(hubs), _ptr(hist))
    return hist


def count_4pcf_parity_hubs(xyz, box_lu, periodic, edges_lu, hubs):
    """Parity-4pCF contribution of the listed hubs (input numbering), no graph."""
    lib = _load()
    xyz, edges, nb, cat = _cat(xyz, box_lu, periodic, edges_lu)
    hubs = np.ascontiguousarray(np.asarray(hubs, dtype=np.int64))
    m = max(nconfig4(nb), 0)
    even = np.zeros(max(m, 1), dtype=np.uint64)
    odd = np.zeros(max(m, 1), dtype=np.int64)
    lib.oracle_4pcf_parity_hubs(*cat, _ptr(hubs), len(hubs), _ptr(even), _ptr(odd))
    return even[:m], odd[:m]


def brute3(xyz, box_lu, periodic, edges_lu) -> np.ndarray:
    lib = _load()
    xyz, edges, nb, cat = _cat(xyz, box_lu, periodic, edges_lu)
    hist = np.zeros(nconfig3(nb), dtype=np.uint64)
    lib.oracle_brute3(*cat, _ptr(hist))
    return hist


def brute4(xyz, box_lu, periodic, edges_lu):
    lib = _load()
    xyz, edges, nb, cat = _cat(xyz, box_lu, periodic, edges_lu)
    m = max(nconfig4(nb), 0)
    even = np.zeros(max(m, 1), dtype=np.uint64)
    odd = np.zeros(max(m, 1), dtype=np.int64)
    lib.oracle_brute4(*cat, _ptr(even), _ptr(odd))
    return even[:m], odd[:m]
