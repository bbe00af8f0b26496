"""ctypes declarations of the C ABI in include/gramsci_gb.h.

Loading fails loudly when libgramsci_gb.so is missing: there is no fallback
implementation of any step.
"""
from __future__ import annotations

import ctypes
import os


_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_int = ctypes.c_int
_p = ctypes.c_void_p

GS_OK, GS_ERR_ARG, GS_ERR_NOMEM, GS_ERR_CUDA, GS_ERR_CAPACITY, GS_ERR_INTERNAL = range(6)
STATUS_NAMES = {0: "GS_OK", 1: "GS_ERR_ARG", 2: "GS_ERR_NOMEM", 3: "GS_ERR_CUDA",
                4: "GS_ERR_CAPACITY", 5: "GS_ERR_INTERNAL"}

# name -> (restype, argtypes); every function the header declares
SIGNATURES = {
    "gs_build_graph": (_int, [_p, _i64, _i64, _int, _i64, _p, _int, _p, ctypes.POINTER(_p)]),
    "gs_build_graph_windowed": (_int, [_p, _i64, _i64, _int, _i64, _p, _int, _i64, _p, ctypes.POINTER(_p)]),
    "gs_graph_windows": (_int, [_p, ctypes.POINTER(_i32), ctypes.POINTER(_i64)]),
    "gs_count_3pcf": (_int, [_p, _p, _i64, _i64, _p]),
    "gs_count3_walk": (_int, [_p]),
    "gs_count_4pcf_parity": (_int, [_p, _p, _p, _i64, _i64, _p]),
    "gs_count_4pcf_parity_static": (_int, [_p, _p, _p, _i64, _i64, _p]),
    "gs_count_3pcf_hubs": (_int, [_p, _p, _i64, _p, _p]),
    "gs_count_2pcf": (_int, [_p, _p, _p]),
    "gs_graph_set_weights": (_int, [_p, _p, _p]),
    "gs_count_2pcf_weighted": (_int, [_p, _p, _p]),
    "gs_count_3pcf_weighted": (_int, [_p, _p, _i64, _i64, _p]),
    "gs_count_4pcf6_weighted": (_int, [_p, _p, _p, _i64, _i64, _p]),
    "gs_count_4pcf6": (_int, [_p, _p, _p, _i64, _i64, _p]),
    "gs_config_count_4pcf6": (_i64, [_int]),
    "gs_config_tuple_4pcf6": (_int, [_int, _i64, _p]),
    "gs_count_4pcf_parity_hubs": (_int, [_p, _p, _i64, _p, _p, _p]),
    "gs_graph_export_rows": (_int, [_p, _p, _i64, _p, _p, _p, _p]),
    "gs_graph_info": (_int, [_p, ctypes.POINTER(_i64), ctypes.POINTER(_i64), ctypes.POINTER(_i32)]),
    "gs_graph_export_csr": (_int, [_p, _p, _p, _p, _p]),
    "gs_graph_export_perm": (_int, [_p, _p, _p]),
    "gs_graph_hub_work": (_int, [_p, _p, _p, _p]),
    "gs_config_count_3pcf": (_i64, [_int]),
    "gs_config_count_4pcf": (_i64, [_int]),
    "gs_config_index_3pcf": (_i64, [_int, _int, _int, _int]),
    "gs_config_index_4pcf": (_i64, [_int, _int, _int, _int]),
    "gs_3pcf_from_host": (_int, [_p, _i64, _i64, _int, _i64, _p, _int, _p, _p]),
    "gs_4pcf_parity_from_host": (_int, [_p, _i64, _i64, _int, _i64, _p, _int, _p, _p, _p]),
    "gs_graph_free": (None, [_p]),
    "gs_last_error": (ctypes.c_char_p, []),
    "gs_version": (ctypes.c_char_p, []),
}



class GraphStats(ctypes.Structure):
    _fields_ = [("n", _i64), ("n_edges", _i64), ("max_degree", _i32), ("max_forward", _i32),
                ("cells_per_axis", _i32), ("reserved", _i32), ("hub_tail", _i64),
                ("spoke_walk", _i64)]


SIGNATURES["gs_graph_stats"] = (_int, [_p, ctypes.POINTER(GraphStats), _p])
SIGNATURES["gs_kernel_launches"] = (ctypes.c_uint64, [])
SIGNATURES["gs_alloc_calls"] = (ctypes.c_uint64, [])
SIGNATURES["gs_measure_smem_atomics"] = (_int, [_int, _int, _int, ctypes.POINTER(ctypes.c_double), _p])

_lib = None


class GramsciError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def lib_path() -> str:
    """The in-tree build, or the file named by GRAMSCI_GB_LIBRARY (another build
    of the same sources, e.g. a debug build)."""
    from . import build as _build
    return os.environ.get("GRAMSCI_GB_LIBRARY") or _build.LIB


def load(build_if_missing: bool = False):
    """The loaded library. Raises if it has not been built (no fallback)."""
    global _lib
    if _lib is None:
        path = lib_path()
        if not os.path.exists(path):
            if build_if_missing:
                from . import build as _build
                _build.build()
            else:
                raise RuntimeError(f"{path} is missing: build it with "
                                   "`python -m cosmology_point_correlation_gb300.build`")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def check(status: int):
    if status != GS_OK:
        raise GramsciError(status, load().gs_last_error().decode())
