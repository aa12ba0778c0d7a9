"""The N > 1 path of bench.py on the CPU: two gloo ranks.

The recurrence shards over independent (batch, head) pairs with no exchange
on the data path, so multi-GPU runs are replicas (weak scaling): every rank
runs its own batch and the job's time is the slowest rank's.  These tests run
bench.py's own aggregation functions in two processes over gloo.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        local_ms = [3.0, 5.0][rank]          # rank 1 is the slow one
        slowest = bench.max_over_ranks(local_ms, device="cpu")
        value = bench.job_throughput(1000, world, slowest)
        seeds = [bench.rank_seed(7, r) for r in range(world)]
        # every rank draws a different batch
        from non_linear_matrix_gb300.inputs import make_inputs
        x = make_inputs(1, 4, 2, 16, 16, "f32", bench.rank_seed(7, rank))
        gathered = [torch.zeros_like(x["v"]) for _ in range(world)]
        dist.all_gather(gathered, x["v"])
        results[rank] = (slowest, value, seeds, bool(torch.equal(gathered[0], gathered[1])))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_the_bench():
    world, port = 2, _free_port()
    with mp.get_context("spawn").Manager() as m:
        results = m.dict()
        mp.start_processes(_worker, args=(world, port, results), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(results)
    for rank in range(world):
        slowest, value, seeds, same_batch = res[rank]
        assert slowest == 5.0                     # max over ranks
        assert value == pytest.approx(2 * 1000 / 5e-3)  # all units / slowest time
        assert seeds[0] != seeds[1]
        assert not same_batch


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(2.5, device="cpu") == 2.5
    assert bench.job_throughput(10, 1, 1.0) == pytest.approx(10_000.0)
