"""The N > 1 bench path runs independent replicas; the only cross-rank step
is the max over ranks of the timings.  Checked here with world_size 2 on the
gloo backend (CPU), as the bench runs it under torchrun."""

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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    mine = [10.0 + rank, 20.0 - rank, 5.0 * (rank + 1)]
    got = bench.max_over_ranks(mine, world, torch.device("cpu"))
    q.put((rank, got, bench.whole_job_rate(32, world, got[0])))
    dist.destroy_process_group()


def test_max_over_ranks_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, rate in out:
        assert got == [11.0, 20.0, 10.0]
        assert rate == pytest.approx(32 * 2 / 11.0e-3)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks([1.0, 2.0], 1, torch.device("cpu")) == [1.0, 2.0]
    assert bench.whole_job_rate(32, 1, 2.0) == pytest.approx(16000.0)
