"""Host logic of bench.py: algorithmic bytes, and the multi-rank aggregation over gloo (world size 2)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from speculative_decode_verify_gdn_gb300.synth import WORKLOADS


def test_algorithmic_bytes_of_the_serving_shape():
    d = WORKLOADS["serve16"].dims
    # per sequence 37,718,016 bytes (state read, 16 states, conv history and snapshots,
    # x, a, b, bf16 outputs) plus 131,328 bytes of per-launch parameters
    assert bench.verify_bytes(d) == 32 * 37_718_016 + 131_328 == 1_207_107_840


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [120.0, 150.0][rank]                       # rank 1 is the slow one
    slowest = bench.max_over_ranks(ms, world)
    value = bench.job_throughput(32 * 16 * 100, world, slowest)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, slowest, value))


def test_two_rank_aggregation_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slowest, value in res:
        assert slowest == 150.0
        assert value == pytest.approx(2 * 32 * 16 * 100 / 0.150)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(10, 1, 1000.0) == 10.0
