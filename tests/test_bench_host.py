"""Host logic of the benchmark: the replica aggregation across ranks (run
as two gloo processes on the CPU), the workload generator and the clock
record parsing."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms_local = [12.0, 20.0][rank]
    ms, value = bench.aggregate(ms_local, 2560, world, dist)
    out[rank] = (ms, value)
    dist.destroy_process_group()


def test_replica_aggregation_two_ranks():
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    for rank in range(2):
        ms, value = out[rank]
        assert ms == 20.0                       # the slowest rank's time
        assert value == pytest.approx(2 * 2560 / 0.020)


def test_single_rank_aggregation():
    import bench
    assert bench.aggregate(8.0, 100, 1) == (8.0, 100 / 0.008)


def test_workload_shapes():
    import bench
    wl = bench.make_workload(256, 10)
    assert wl["n_flag"] == 26 and wl["n_ver"] * wl["window"] == 256
    assert wl["ctx"].min() >= 4 and wl["ctx"].max() <= 2048 + 1024
    # same seed, same workload
    wl2 = bench.make_workload(256, 10)
    assert np.array_equal(wl["ctx"], wl2["ctx"])
