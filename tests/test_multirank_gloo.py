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
