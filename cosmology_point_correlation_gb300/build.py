"""Build libgramsci_gb.so (all CUDA sources, sm_103a only) in the package directory.

Each .cu file is compiled by its own nvcc process in parallel, then linked
into one shared library with the C ABI of include/gramsci_gb.h. The checked
variant, libgramsci_gb_checked.so, is the same sources compiled with
-DGS_CHECKED: its hot kernels test their memory indices and the calls report
GS_ERR_INTERNAL when a test fails (tests load it through GRAMSCI_GB_LIBRARY).
"""
from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libgramsci_gb.so")
CHECKED_LIB = os.path.join(PKG, "libgramsci_gb_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgramsci_gb.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + \
        sorted(glob.glob(os.path.join(INCLUDE, "*.h"))) + [os.path.abspath(__file__)]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def _build_jobs(checked: bool):
    """(library, object directory, extra flags) of one variant."""
    if checked:
        return CHECKED_LIB, os.path.join(BUILD_DIR, "checked"), ["-DGS_CHECKED"]
    return LIB, BUILD_DIR, []


def build(force: bool = False, verbose: bool = False, checked: bool | None = None) -> str:
    """Build the library (checked=False), its checked variant (True) or both
    (None, the default; the two compile in parallel). Returns the regular
    library's path (the checked one's when checked=True)."""
    variants = [False, True] if checked is None else [checked]
    todo = [v for v in variants if force or not up_to_date(_build_jobs(v)[0])]
    if todo:
        cc = nvcc()
        for v in todo:
            os.makedirs(_build_jobs(v)[1], exist_ok=True)

        def compile_one(job):
            v, src = job
            _, objdir, extra = _build_jobs(v)
            obj = os.path.join(objdir, os.path.basename(src) + ".o")
            cmd = [cc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
            return v, obj, r.stderr

        jobs = [(v, src) for v in todo for src in _sources()]
        with concurrent.futures.ThreadPoolExecutor(max_workers=min(16, len(jobs))) as ex:
            results = list(ex.map(compile_one, jobs))
        if verbose:
            for _, _, log in results:
                print(log)
        for v in todo:
            lib = _build_jobs(v)[0]
            tmp = lib + f".{os.getpid()}.tmp"
            cmd = [cc, *ARCH, "-shared", "-o", tmp] + [o for w, o, _ in results if w == v]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
            os.replace(tmp, lib)
    return CHECKED_LIB if checked else LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
