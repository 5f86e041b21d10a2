"""Host logic of bench.py's multi-rank path on CPU: two gloo ranks report different step
times; the job time is the slowest rank's and the job throughput counts both ranks' work."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    my_ms = 100.0 + 50.0 * rank
    mx = bench.reduce_max(my_ms, dist)
    out[rank] = mx
    out[world + rank] = bench.job_throughput(4e12, 10, world, mx)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_max_time():
    world, port = 2, _free_port()
    out = torch.zeros(2 * world, dtype=torch.float64).share_memory_()
    mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1] == 150.0
    assert out[2] == out[3] == pytest.approx(2 * 4e12 * 10 / 0.150 / 1e12)


def test_single_rank_is_identity():
    assert bench.reduce_max(12.5, None) == 12.5
    assert bench.job_throughput(4e12, 10, 1, 100.0) == pytest.approx(400.0)


def test_call_stats_percentiles():
    """The per-call distribution: 50 calls in 5 rounds, percentiles by linear interpolation
    (numpy's default rule), min/max/mean exact."""
    import numpy as np
    rounds = [[float(10 * r + i) for i in range(10)] for r in range(5)]   # 0..49
    st = bench.call_stats(rounds)
    xs = np.arange(50, dtype=np.float64)
    assert st["count"] == 50 and st["min"] == 0.0 and st["max"] == 49.0
    assert st["mean"] == pytest.approx(24.5)
    for q in (50, 90, 95, 99):
        assert st[f"p{q}"] == pytest.approx(float(np.percentile(xs, q)), abs=1e-4)
    assert st["round_means"] == [4.5, 14.5, 24.5, 34.5, 44.5]
    assert bench.call_stats([[3.0]])["p90"] == 3.0
