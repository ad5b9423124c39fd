"""The benchmark's multi-rank arithmetic on CPU: two gloo ranks each time their
own replica; the whole-job value divides all ranks' tokens by the slowest rank's
time (max over ranks), and no data crosses ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, l = bench.dist_env()
    assert (w, r, l) == (world, rank, rank)
    secs = [2.0, 3.0][rank]          # rank 1 is the slow one
    value, tmax = bench.whole_job_value(1000.0, secs, world)
    q.put((rank, value, tmax))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_whole_job_value_uses_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for _, value, tmax in res:
        assert tmax == pytest.approx(3.0)
        assert value == pytest.approx(2 * 1000.0 / 3.0)


def test_single_rank_is_identity():
    import bench
    assert bench.whole_job_value(500.0, 2.0, 1) == (250.0, 2.0)
