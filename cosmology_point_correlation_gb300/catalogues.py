"""Seeded synthetic point catalogues on the 1/1024 h^-1 Mpc integer lattice.

This module only draws random numbers and quantises them. It holds none of the
counting method's arithmetic (no distances, bins or determinants), so both the
CUDA path and the CPU oracle can take their inputs from it.

Two point processes stand in for the catalogues the GRAMSCI v2 paper
("Fast Graph-based Higher-Order Clustering Statistics on the GPU") measures on:
uniform randoms (§IV.1 test catalogue randoms) and a Neyman-Scott cluster
process standing in for clustered galaxy samples with a heavy-tailed neighbour
count distribution (§V.2, the <m^3> >> <m>^3 remark).

Quantisation: a float position x (h^-1 Mpc) becomes floor(x * 1024) mod Lu
with Lu = round(L * 1024), stored as int32. Cluster offsets are wrapped into
the box for every catalogue, periodic or not, so N and the mean density are
exactly as requested.
"""
from __future__ import annotations

import numpy as np

LATTICE_PER_MPC = 1024


def box_lattice(box_mpc: float) -> int:
    """Box side in lattice units."""
    return int(round(box_mpc * LATTICE_PER_MPC))


def _quantise(x_mpc: np.ndarray, box_lu: int) -> np.ndarray:
    q = np.floor(x_mpc * LATTICE_PER_MPC).astype(np.int64) % box_lu
    return np.ascontiguousarray(q.astype(np.int32))


def uniform(n: int, box_mpc: float, seed: int) -> np.ndarray:
    """n points with iid uniform integer lattice coordinates in [0, Lu)^3."""
    lu = box_lattice(box_mpc)
    rng = np.random.Generator(np.random.PCG64(seed))
    return np.ascontiguousarray(rng.integers(0, lu, size=(n, 3), dtype=np.int64).astype(np.int32))


def neyman_scott(n: int, box_mpc: float, n_parents: int, mu: float, sigma_mpc: float,
                 seed: int) -> np.ndarray:
    """n points from a Neyman-Scott process.

    Parent centres are uniform in the box. Each parent gets Poisson(mu)
    children with iid N(0, sigma^2) offsets per axis, wrapped into the box.
    Clusters are appended one parent at a time until the catalogue holds n
    points; the last cluster is cut at exactly n. The number of parents used
    is therefore n_parents = n / mu in expectation.
    """
    if n <= 0:
        return np.zeros((0, 3), dtype=np.int32)
    lu = box_lattice(box_mpc)
    rng = np.random.Generator(np.random.PCG64(seed))
    # Draw more parents than needed; only a prefix is used.
    cap = max(2 * n_parents, 16)
    while True:
        counts = rng.poisson(mu, size=cap)
        if counts.sum() >= n:
            break
        cap *= 2
    csum = np.cumsum(counts)
    used = int(np.searchsorted(csum, n)) + 1        # parents needed to reach n points
    counts = counts[:used].copy()
    counts[-1] -= int(csum[used - 1] - n)            # cut the last cluster at exactly n
    parents = rng.uniform(0.0, box_mpc, size=(used, 3))
    offsets = rng.normal(0.0, sigma_mpc, size=(n, 3))
    pos = np.repeat(parents, counts, axis=0) + offsets
    pos = np.mod(pos, box_mpc)
    return _quantise(pos, lu)


def linear_edges_lu(r_max_mpc: float, nbins: int, r_min_mpc: float = 0.0) -> np.ndarray:
    """nbins+1 linear bin edges in lattice units, rounded to the nearest lattice step."""
    e = np.linspace(r_min_mpc, r_max_mpc, nbins + 1) * LATTICE_PER_MPC
    return np.ascontiguousarray(np.rint(e).astype(np.int64))
