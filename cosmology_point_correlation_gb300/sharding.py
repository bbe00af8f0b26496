"""Hub ranges and the histogram reduction for splitting one graph's counts
across processes.

Hubs are independent units of the counts (the GRAMSCI v2 paper, §IV.7: tiles
partition the work by hub window with no communication), so contiguous hub
ranges in the graph's internal order can go to different ranks and their
integer histograms add exactly. This module computes the ranges (balanced on
the per-hub merge-walk work the library exports) and sums the ranks'
histograms; the counts themselves run in the library on each rank.
"""
from __future__ import annotations

import numpy as np

# per-hub cost of a 3pCF count beyond its walk: staging the hub's row and
# handing out its spokes, in units of spoke-row entries walked
HUB_OVERHEAD = 64


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
        cuts = np.searchsorted(c, targets, side="left").clip(0, n)
        # the nearer of the two prefix sums around each target
        lower = (cuts - 1).clip(0, n)
        cuts = np.where((cuts > 0) & (targets - c[lower] < c[cuts] - targets), lower, cuts).tolist()
        cuts[0], cuts[-1] = 0, n
        for r in range(1, world + 1):
            cuts[r] = max(cuts[r], cuts[r - 1])
    return [(int(cuts[r]), int(cuts[r + 1])) for r in range(world)]


def count3_work(fwd, walk):
    """Per-hub work of the 3pCF count from the library's hub work export
    (Graph.hub_work): the spoke-row entries the hub's merge-walks read, plus
    its forward row and a fixed per-hub cost."""
    return np.asarray(walk, dtype=np.float64) + np.asarray(fwd, dtype=np.float64) + HUB_OVERHEAD


def balanced_ranges(fwd, walk, world: int):
    """Contiguous hub ranges of about equal 3pCF work, one per rank."""
    return hub_ranges(len(fwd), world, count3_work(fwd, walk))


def reduce_histograms(*hists):
    """Sum each int64 histogram tensor over all ranks, in place (the counts are
    integers, so the sum is exact and independent of the order of ranks).
    uint64 counts held in int64 tensors add the same way bit for bit."""
    import torch.distributed as dist
    for h in hists:
        dist.all_reduce(h, op=dist.ReduceOp.SUM)
    return hists
