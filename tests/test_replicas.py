"""The multi-GPU bench path runs independent replicas: the step time is the
slowest rank's, the throughput counts every rank's units. Checked here with
two gloo ranks on the CPU (no GPU, no collective on any data path)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out):
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [3.0, 5.0][rank]                      # rank 1 is the slower replica
        ms = bench.max_over_ranks(local_ms, dist, "cpu")
        rate = bench.whole_job_rate(1, world, ms * 1e-3)
        out.put((rank, ms, rate))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_count_all_units():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [5.0, 5.0]
    # 1 token per rank per step, 2 ranks, 5 ms per step: 400 tokens/s
    assert all(abs(r[2] - 400.0) < 1e-9 for r in res)


def test_single_process_needs_no_group():
    import bench
    assert bench.max_over_ranks(2.5) == 2.5
    assert bench.whole_job_rate(16, 1, 0.002) == 8000.0



def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    import argparse
    import bench
    monkeypatch.setenv("RANK", "1")
    args = argparse.Namespace(config=0, tokens=None, layers=None, steps=1, warmup=0, gpus=2)
    assert bench.run_reference(args) == 0            # returns at once, prints nothing
