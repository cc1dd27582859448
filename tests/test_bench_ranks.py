"""The bench's multi-rank path (one independent replica per GPU, no
collective on the data path): the job time is the slowest rank's and the job
value counts every rank's bytes.  Two gloo ranks on the CPU."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [120.0, 150.0][rank]
    total = bench.max_over_ranks(local_ms, world)
    value = bench.job_value(1_000_000_000, world, 10, total)
    torch.distributed.barrier()
    torch.distributed.destroy_process_group()
    out[rank] = (total, value)


def test_two_rank_max_time_and_job_value():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = free_port()
    procs = [ctx.Process(target=worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        total, value = out[r]
        assert total == 150.0
        assert value == pytest.approx(1e9 * 2 * 10 / 0.150 / 1e9)


def test_single_rank_passthrough():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_value(2_000_000_000, 1, 4, 1000.0) == pytest.approx(8.0)
