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
    assert wl["n_flag"] == 26 and wl["groups"] == [4, 8, 16]
    assert wl["max_window"] == 64 and wl["headroom"] >= 64
    assert wl["ctx"].min() >= 4 and wl["ctx"].max() <= 2048 + 1024
    # same seed, same workload
    wl2 = bench.make_workload(256, 10)
    assert np.array_equal(wl["ctx"], wl2["ctx"])


def test_verify_plans_layout_and_expected_commits():
    """The bench's verify plans: group sizes cycle over 4 / 8 / 16 with
    windows of 64 / 32 / 16 candidates (256 rows each), the requests of a
    plan are distinct flagged requests, the plan array holds the windows in
    the device layout (count, requests, contexts, last tokens, lengths,
    candidates), and the expected commit is the first perturbed index."""
    import bench
    from deterministic_invariant_bf16_gb300 import binding as bi
    wl = bench.make_workload(256, 10)
    V = 128256
    rng = np.random.default_rng(0)
    greedy = rng.integers(0, V, size=(wl["n_flag"], wl["max_window"]))
    plans, expect, meta = bench.verify_plans(wl, greedy, V, n_plans=12)
    n = bi.VERIFY_ROWS
    flips = 0
    for k, (a, exp, m) in enumerate(zip(plans, expect, meta)):
        g = [4, 8, 16][k % 3]
        assert m["g"] == g and m["w"] * g == 256
        assert len(set(m["reqs"])) == g
        assert all(0 <= r < wl["n_flag"] for r in m["reqs"])
        assert a[0] == g
        assert list(a[8:8 + g]) == m["reqs"]
        assert list(a[8 + n:8 + n + g]) == [int(wl["ctx"][r])
                                            for r in m["reqs"]]
        assert list(a[8 + 2 * n:8 + 2 * n + g]) == [
            int(wl["first_tokens"][r]) for r in m["reqs"]]
        assert all(a[8 + 3 * n:8 + 3 * n + g] == m["w"])
        cands = a[8 + 4 * n:8 + 5 * n]
        for i, (r, win, j) in enumerate(zip(m["reqs"], m["windows"], exp)):
            assert list(cands[i * m["w"]:(i + 1) * m["w"]]) == win
            diff = np.nonzero(np.array(win) != greedy[r][:m["w"]])[0]
            assert j == (diff[0] if len(diff) else m["w"])
            flips += len(diff)
    assert flips > 0   # some windows roll back
