"""The multi-rank host logic of bench.py on CPU: two gloo ranks (127.0.0.1), each with
its own timing; the job time is the slowest rank's and the job throughput counts every
rank's work (independent replicas, no data-path collective)."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        local = [10.0 + rank, 5.0 - rank, 7.0 * (rank + 1)]  # ms: step, kernel, e2e
        got = bench.max_over_ranks(local, dist, "cpu")
        out[rank] = got + [bench.job_tflops(world, 2.0e12, got[0])]
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_sum_the_work():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        step, kern, e2e, tflops = res[r]
        assert step == 11.0 and kern == 5.0 and e2e == 14.0
        # 2 ranks x 2 TFLOP in 11 ms
        assert tflops == pytest.approx(2 * 2.0e12 / 11e-3 / 1e12)


def test_single_process_is_the_identity():
    import bench
    assert bench.max_over_ranks([1.5, 2.5], None, "cpu") == [1.5, 2.5]
    assert bench.job_tflops(1, 1e12, 1000.0) == pytest.approx(1.0)
