"""The multi-process path on CPU (gloo, world size 2): hub ranges balanced on
the per-hub merge-walk work split one count across ranks, and the integer
histograms all-reduce (with the reduction bench.py --strong uses) to the full
one; the benchmark's cross-rank reduction of timings takes the max of times
and the sum of counts."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from cosmology_point_correlation_gb300 import catalogues
from cosmology_point_correlation_gb300.sharding import balanced_ranges, hub_ranges, reduce_histograms


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, result):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        box = 30000
        xyz = catalogues.neyman_scott(600, box / 1024, 12, 50.0, 1.5, 17)
        edges = catalogues.linear_edges_lu(5.0, 5)
        g = oracle.graph(xyz, box, 1, edges)
        # the per-hub work the library's hub_work export gives: forward degree
        # f_i and the spoke-row entries w_i = sum of f_j over forward spokes j
        n = len(xyz)
        fwd = np.array([(g.nbr[g.row_ptr[i]:g.row_ptr[i + 1]] > i).sum() for i in range(n)])
        walk = np.array([fwd[[j for j in g.nbr[g.row_ptr[i]:g.row_ptr[i + 1]] if j > i]].sum()
                         for i in range(n)])
        b, e = balanced_ranges(fwd, walk, world)[rank]
        h3 = torch.from_numpy(oracle.count_3pcf(xyz, box, 1, edges, g, b, e).astype(np.int64))
        ev, od = oracle.count_4pcf_parity(xyz, box, 1, edges, g, b, e)
        h4 = torch.from_numpy(np.concatenate([ev.astype(np.int64), od]))
        reduce_histograms(h3, h4)                 # the reduction bench.py --strong uses
        import bench
        mx, sm = bench.reduce_max_sum(world, [float(rank + 1), 10.0 * rank], [float(rank + 1)])
        if rank == 0:
            full3 = oracle.count_3pcf(xyz, box, 1, edges, g).astype(np.int64)
            fe, fo = oracle.count_4pcf_parity(xyz, box, 1, edges, g)
            result["ok3"] = bool(np.array_equal(h3.numpy(), full3))
            result["ok4"] = bool(np.array_equal(h4.numpy(), np.concatenate([fe.astype(np.int64), fo])))
            result["max"] = mx
            result["sum"] = sm
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reproduce_the_full_counts():
    world = 2
    with mp.Manager() as man:
        result = man.dict()
        mp.spawn(_worker, args=(world, _free_port(), result), nprocs=world, join=True)
        assert result["ok3"] and result["ok4"]
        assert result["max"] == [2.0, 10.0]
        assert result["sum"] == [3.0]


def test_hub_ranges_cover_and_balance():
    assert hub_ranges(10, 3) == [(0, 3), (3, 6), (6, 10)]
    assert hub_ranges(0, 2) == [(0, 0), (0, 0)]
    w = np.array([100, 1, 1, 1, 1, 1, 1, 1, 1, 1], dtype=float)
    r = hub_ranges(10, 2, w)
    assert r[0][0] == 0 and r[-1][1] == 10 and r[0][1] == r[1][0]
    assert r[0] == (0, 1)
    with pytest.raises(ValueError):
        hub_ranges(5, 0)


def test_balanced_ranges_follow_the_walk_work():
    fwd = np.array([0, 5, 5, 0, 0, 0, 0, 0])
    walk = np.array([0, 1000, 1000, 0, 0, 0, 0, 0])
    r = balanced_ranges(fwd, walk, 2)
    assert r[0][0] == 0 and r[-1][1] == 8 and r[0][1] == r[1][0]
    assert r[0][1] == 2                      # the two heavy hubs go to different ranks


def test_hub_ranges_properties_on_random_work():
    # Every cut is the nearer of the two prefix sums around its target, so it
    # lies within half the largest hub weight of the target, and each range's
    # work within one largest weight of total / world; the ranges are
    # contiguous, ordered and cover [0, n) for any world size.
    rng = np.random.default_rng(7)
    for trial in range(300):
        n = int(rng.integers(0, 60))
        world = int(rng.integers(1, 12))
        kind = trial % 3
        if kind == 0:
            w = rng.integers(0, 1000, size=n).astype(float)
        elif kind == 1:                                 # heavy tail, many empty hubs
            w = np.where(rng.random(n) < 0.5, 0.0, rng.pareto(1.2, size=n) * 100).round()
        else:                                           # one dominant hub
            w = np.ones(n)
            if n:
                w[int(rng.integers(0, n))] = 10_000.0
        r = hub_ranges(n, world, w)
        assert len(r) == world
        assert r[0][0] == 0 and r[-1][1] == n
        for (b0, e0), (b1, e1) in zip(r, r[1:]):
            assert e0 == b1
        assert all(b <= e for b, e in r)
        if n == 0:
            continue
        share, wmax = w.sum() / world, w.max()
        for b, e in r:
            assert abs(w[b:e].sum() - share) <= wmax + 1e-9 * max(1.0, w.sum())
        # without weights the sizes differ by at most one hub
        sizes = [e - b for b, e in hub_ranges(n, world)]
        assert max(sizes) - min(sizes) <= 1 and sum(sizes) == n
