"""The multi-process path on CPU (gloo, world size 2): hub ranges split one
count across ranks and the integer histograms all-reduce to the full one; the
benchmark's cross-rank reduction takes the max of times and the sum of counts."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from cosmology_point_correlation_gb300 import catalogues
from cosmology_point_correlation_gb300.sharding import hub_ranges


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
        deg = np.diff(g.row_ptr)
        b, e = hub_ranges(len(xyz), world, weights=deg.astype(np.float64) ** 2)[rank]
        h3 = torch.from_numpy(oracle.count_3pcf(xyz, box, 1, edges, g, b, e).astype(np.int64))
        ev, od = oracle.count_4pcf_parity(xyz, box, 1, edges, g, b, e)
        h4 = torch.from_numpy(np.concatenate([ev.astype(np.int64), od]))
        dist.all_reduce(h3)
        dist.all_reduce(h4)
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
