"""The checked build (libgramsci_gb_checked.so: the sources compiled with
GS_CHECKED, whose graph build, 3pCF and parity kernels test the indices of
their memory accesses and make the call fail with GS_ERR_INTERNAL when a test
fails) runs the small GPU cases with every result equal to the oracle's and
no failed check. It runs in a process of its own, since a process loads one
build of the library."""
import os
import subprocess
import sys

import pytest

from cosmology_point_correlation_gb300 import build

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checked_build_runs_clean():
    lib = build.build(checked=True)
    env = dict(os.environ, GRAMSCI_GB_LIBRARY=lib)
    r = subprocess.run([sys.executable, "-m", "tests.checked_run"], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "no device check failed" in r.stdout
