"""The bench's multi-rank logic on CPU: two gloo ranks, each timing its own
sequences (weak scaling). The job's step time is the slowest rank's, and the
whole-job throughput counts every rank's sequences."""
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


def _rank(rank, world, port, out):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [12.5, 20.0][rank]          # rank 1 is the slower one
        ms = bench.max_over_ranks(local_ms, world, "cpu")
        dist.barrier()
        out[rank] = (ms, bench.job_tokens_per_s(world, 4, ms / 10))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_time_and_job_throughput():
    port = _free_port()
    out = mp.Manager().dict()
    mp.start_processes(_rank, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert out[0] == out[1]
    ms, tps = out[0]
    assert ms == pytest.approx(20.0)
    # 2 ranks x 4 sequences, one token each per 2 ms step
    assert tps == pytest.approx(2 * 4 * 1000.0 / 2.0)


def test_single_rank_is_local():
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.job_tokens_per_s(1, 4, 0.5) == pytest.approx(8000.0)
