"""The multi-rank path of bench.py on CPU: two gloo ranks (processes) run
the same reduction the benchmark runs over its GPUs -- the job's time is the
slowest rank's, and its throughput counts every rank's tokens (independent
replicas, weak scaling)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    dev = torch.device("cpu")
    dist.barrier()
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, world, dev)   # rank 1 is the slow one
    e2e = bench.max_over_ranks(0.5 * (world - rank), world, dev)
    value = bench.job_tokens_per_s(765, 4, world, ms)
    out[rank] = (ms, e2e, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_count_all_tokens():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        ms, e2e, value = res[r]
        assert ms == 15.0 and e2e == 1.0
        assert value == pytest.approx(765 * 4 * 2 / 0.015)


def test_single_rank_is_unchanged():
    import bench
    assert bench.max_over_ranks(3.25, 1, torch.device("cpu")) == 3.25
    assert bench.job_tokens_per_s(100, 10, 1, 1000.0) == pytest.approx(1000.0)
