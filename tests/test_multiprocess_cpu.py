"""Replica timing logic of bench.py over two gloo ranks on the CPU: every
rank runs its own batch (no data-path collective); the only cross-rank steps
are the barrier and the max over ranks of the elapsed time."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    from workloads import OLMOE
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        dist.barrier()
        my_ms = 100.0 + 25.0 * rank           # the slower rank decides
        total = bench.max_over_ranks(my_ms, dist, "cpu")
        out[rank] = (total, bench.rank_seed(OLMOE, rank),
                     bench.aggregate_tokens_per_s(OLMOE.n, 20, world, total))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_distinct_batches():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    from workloads import OLMOE
    assert res[0][0] == res[1][0] == 125.0
    assert res[0][1] == OLMOE.seed and res[1][1] != OLMOE.seed
    assert res[0][2] == pytest.approx(2 * 4096 * 20 / 0.125)


def test_single_process_needs_no_collective():
    import bench
    assert bench.max_over_ranks(3.5, None) == 3.5
    assert bench.aggregate_tokens_per_s(4096, 10, 1, 5.0) == pytest.approx(4096 * 10 / 0.005)
