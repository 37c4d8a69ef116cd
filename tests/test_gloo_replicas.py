"""The N-GPU bench runs N independent replicas; its only cross-rank steps are
the barrier and the max over ranks of the step time. Checked here with two
gloo ranks on the CPU (no GPU involved)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    import sys
    import torch.distributed as dist
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    step_ms = [0.25, 0.40][rank]
    slowest = bench.max_over_ranks(step_ms)
    dist.barrier()
    results[rank] = (slowest, bench.job_tokens_per_s(4096, world, slowest))
    dist.destroy_process_group()


def test_two_rank_aggregation_takes_the_slowest_rank():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    results = mgr.dict()
    mp.start_processes(_rank, args=(world, port, results), nprocs=world, join=True,
                       start_method="spawn")
    for r in range(world):
        slowest, tps = results[r]
        assert slowest == pytest.approx(0.40)
        assert tps == pytest.approx(2 * 4096 / 0.40e-3)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(1.5) == 1.5
    assert bench.job_tokens_per_s(4096, 1, 2.0) == pytest.approx(4096 / 2e-3)
