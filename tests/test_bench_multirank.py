"""bench.py's multi-rank bookkeeping on CPU with two gloo ranks: the step time is the slowest
replica's and the value counts every rank's tokens (no GPU involved)."""
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


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = bench.slowest_replica_ms(1.0 + 2.5 * rank, world, torch.device("cpu"))
        q.put((rank, ms, bench.job_tokens(16384, world)))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_take_the_slowest_and_count_all_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=90) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [3.5, 3.5]          # max over ranks on every rank
    assert [g[2] for g in got] == [32768, 32768]      # whole-job tokens


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.slowest_replica_ms(2.0, 1, torch.device("cpu")) == 2.0
    assert bench.job_tokens(100, 1) == 100
