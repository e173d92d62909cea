"""The bench's multi-rank path on CPU: two gloo ranks, each reporting its own
timed region; the job throughput is all ranks' events over the slowest rank's
time (weak scaling, no data-path collective)."""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [40.0, 50.0][rank]  # rank 1 is the slower one
    value, ms = bench.job_throughput(local_ms, events_per_rank=320, world=world, dist=dist, device="cpu")
    out[rank] = (value, ms)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_weak_scaling():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        value, ms = out[r]
        assert ms == pytest.approx(50.0)
        assert value == pytest.approx(2 * 320 / 0.050)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    value, ms = bench.job_throughput(25.0, events_per_rank=32, world=1)
    assert ms == 25.0 and value == pytest.approx(32 / 0.025)
