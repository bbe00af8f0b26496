"""The C ABI loads and exports every function include/*.h declares; the
host-only entry points work without a GPU. CPU only: no compute call here
touches a device."""
import glob
import os
import re

import numpy as np
import pytest

from cosmology_point_correlation_gb300 import _lib, build
from tests import fixtures as fx

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(gs_[a-z0-9_]+)\s*\(", text))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert {"gs_build_graph", "gs_count_3pcf", "gs_count_4pcf_parity"} <= names
    for n in sorted(names):
        assert hasattr(lib, n), n
    assert names == set(_lib.SIGNATURES), "binding and header disagree"


def test_config_counts(lib):
    assert lib.gs_config_count_3pcf(10) == 220      # GRAMSCI v2 §V.1: 220 configurations, 10 bins
    for nb in range(1, 40):
        assert lib.gs_config_count_3pcf(nb) == len(fx.configs3(nb))
        assert lib.gs_config_count_4pcf(nb) == len(fx.configs4(nb))
    assert lib.gs_config_count_3pcf(0) == -1 and lib.gs_config_count_3pcf(256) == -1


@pytest.mark.parametrize("nb", [1, 2, 3, 5, 8, 15, 30, 41])
def test_config_index_matches_enumeration(lib, nb):
    for k, c in enumerate(fx.configs3(nb)):
        assert lib.gs_config_index_3pcf(nb, *c) == k
    for k, c in enumerate(fx.configs4(nb)):
        assert lib.gs_config_index_4pcf(nb, *c) == k
    assert lib.gs_config_index_3pcf(nb, 1, 0, 0) == -1
    assert lib.gs_config_index_4pcf(nb, 0, 0, 1) == -1


def test_version_and_error_string(lib):
    assert b"sm_103a" in lib.gs_version()
    assert isinstance(lib.gs_last_error(), bytes)


def test_null_graph_is_rejected_without_device_work(lib):
    assert lib.gs_graph_info(None, None, None, None) == _lib.GS_ERR_ARG
    assert b"NULL" in lib.gs_last_error()
    lib.gs_graph_free(None)


def test_3pcf_slices_follow_the_configuration_order(lib):
    from cosmology_point_correlation_gb300 import equilateral, isosceles, xi_natural
    nb = 7
    cfg = fx.configs3(nb)
    hist = np.arange(len(cfg))              # entry k holds k
    assert equilateral(hist, nb).tolist() == [cfg.index((b, b, b)) for b in range(nb)]
    assert isosceles(hist, nb, 3).tolist() == [cfg.index(tuple(sorted((3, 3, c)))) for c in range(nb)]
    xi = xi_natural([10, 0], [10, 5], 101, 101)
    assert xi[0] == 0.0 and xi[1] == -1.0


def test_six_bin_configuration_tuples_and_disconnected_term(lib):
    import oracle
    from cosmology_point_correlation_gb300 import config_tuples_4pcf6, zeta4_disconnected
    assert lib.gs_config_count_4pcf6(4) == 276 and lib.gs_config_count_4pcf6(11) == -1
    t = config_tuples_4pcf6(4)
    assert t.shape == (276, 6)
    for k in range(0, 276, 7):              # the oracle's own enumeration agrees
        assert oracle.config_index6(4, t[k]) == k
    xi = np.array([0.5, 0.25, 0.125, 0.0625])
    z = zeta4_disconnected(xi, 4)
    k = oracle.config_index6(4, (0, 1, 2, 2, 2, 3))
    # pairings (01,23), (02,13), (03,12): xi0*xi3 + xi1*xi2 + xi2*xi2
    assert z[k] == xi[0] * xi[3] + xi[1] * xi[2] + xi[2] * xi[2]
    # Eq.(4) is the same for every labelling of a tetrahedron
    k0 = oracle.config_index6(4, (0, 0, 0, 0, 0, 0))
    assert z[k0] == 3 * xi[0] ** 2


def test_signed_xi_and_connected_four_point(lib):
    import oracle
    from cosmology_point_correlation_gb300 import as_int128, xi_signed, zeta4_connected, zeta4_disconnected
    # 128-bit (low, high) words back to integers, signs included
    words = np.array([[5, 0], [-1, -1], [0, 1], [-(1 << 63), 7]], dtype=np.int64)
    assert as_int128(words) == [5, -1, 1 << 64, (7 << 64) + (1 << 63)]
    # xi = signed pair sum / RR (Eq.(5)'s xi, §III.3)
    assert xi_signed([3, -2, 0], [6, 8, 5]).tolist() == [0.5, -0.25, 0.0]
    # zeta_conn = NNNN / RRRR - zeta_disc(xi), per configuration
    xi = np.array([0.5, 0.25, 0.125, 0.0625])
    rrrr = [1 << 70] * 276
    nnnn = [(k + 1) << 66 for k in range(276)]
    zc = zeta4_connected(nnnn, rrrr, xi, 4)
    k = oracle.config_index6(4, (0, 1, 2, 2, 2, 3))
    assert zc[k] == (k + 1) / 16 - (xi[0] * xi[3] + xi[1] * xi[2] + xi[2] * xi[2])
    assert np.allclose(zc + zeta4_disconnected(xi, 4), [(k + 1) / 16 for k in range(276)], rtol=0, atol=0)
