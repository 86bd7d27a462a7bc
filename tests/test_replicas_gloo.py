"""The N > 1 path of the benchmark, on CPU with gloo, world size 2: each rank
is an independent replica (no data-path collective); the only cross-rank
step is the host-side max of the timings, and the whole-job throughput counts
every rank's batch."""
import os
import socket

import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [10.0 + rank, 5.0 - rank]      # region ms, launch ms of this rank
        got = bench.max_over_ranks(mine, world)
        dist.barrier()
        results[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_ranks():
    world = 2
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), results), nprocs=world, join=True)
        assert results[0] == [11.0, 5.0] and results[1] == [11.0, 5.0]


def test_whole_job_throughput_counts_every_replica():
    # 2 ranks x 1024 tokens x 100 steps in 50 ms (the slowest rank's time).
    assert bench.whole_job_tokens_per_s(2, 1024, 100, 50.0) == 2 * 1024 * 100 / 0.05
    assert bench.max_over_ranks([3.0, 4.0], 1) == [3.0, 4.0]
