"""Hub ranges for splitting one graph's counts across processes.

Hubs are independent units of the counts (the GRAMSCI v2 paper, §IV.7: tiles
partition the work by hub window with no communication), so contiguous hub
ranges in the graph's internal order can go to different ranks and their
integer histograms add exactly. This module only computes the ranges; the
counts themselves run in the library on each rank.
"""
from __future__ import annotations

import numpy as np


def hub_ranges(n: int, world: int, weights=None):
    """`world` contiguous [begin, end) ranges covering [0, n).

    Without weights the ranges hold equal numbers of hubs; with per-hub work
    weights (length n, non-negative) each range holds about 1/world of the
    total weight.
    """
    if world < 1:
        raise ValueError("world must be >= 1")
    if weights is None:
        cuts = [(n * r) // world for r in range(world + 1)]
    else:
        w = np.asarray(weights, dtype=np.float64)
        if w.shape != (n,) or np.any(w < 0):
            raise ValueError("weights must be n non-negative numbers")
        c = np.concatenate([[0.0], np.cumsum(w)])
        targets = c[-1] * np.arange(world + 1) / world
        cuts = np.searchsorted(c, targets, side="left").clip(0, n).tolist()
        cuts[0], cuts[-1] = 0, n
        for r in range(1, world + 1):
            cuts[r] = max(cuts[r], cuts[r - 1])
    return [(int(cuts[r]), int(cuts[r + 1])) for r in range(world)]
