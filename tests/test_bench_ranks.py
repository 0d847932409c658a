"""The multi-rank host logic of bench.py on CPU: two gloo ranks, each with its
own timings, must both see the per-value maximum, and the whole-job rate must
count every rank's work against the slowest rank's time."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r: step 1 + r ms, end-to-end 5 - r ms, launch 2 ms
        got = bench.max_over_ranks([1.0 + rank, 5.0 - rank, 2.0], dist)
        out.put((rank, got))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert results == {0: [2.0, 5.0, 2.0], 1: [2.0, 5.0, 2.0]}


def test_max_over_ranks_without_a_group_is_identity():
    import torch.distributed as dist
    assert bench.max_over_ranks([3, 1.5], None) == [3.0, 1.5]
    if not dist.is_initialized():
        assert bench.max_over_ranks([3, 1.5], dist) == [3.0, 1.5]


@pytest.mark.parametrize("world", [1, 2, 8])
def test_whole_job_rate_counts_all_ranks(world):
    # 268,435,456 bytes per rank in 0.05 ms on the slowest rank
    v = bench.whole_job_rate(world, 268435456, 0.05, 1e9)
    assert v == pytest.approx(world * 268435456 / 0.05e-3 / 1e9)
