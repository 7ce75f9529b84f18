"""The N > 1 timing path of the benchmark on CPU: two gloo ranks, each a
replica with its own timed region; the job time is the slowest rank's and
the throughput counts both replicas' bytes."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        dist.barrier()
        t_local = 1.0 + rank          # rank 1 is the slow one
        t = bench.slowest_rank_time(t_local, world, device="cpu")
        v = bench.job_throughput(bytes_per_step=1e9, steps=4, world=world, t=t)
        dist.barrier()
        out[rank] = (t, v)
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(90)
        assert p.exitcode == 0
    for r in range(2):
        t, v = out[r]
        assert t == 2.0                       # max over ranks
        assert abs(v - 1e9 * 4 * 2 / 2.0 / 1e9) < 1e-9   # both replicas' bytes


def test_single_rank_is_identity():
    import bench
    assert bench.slowest_rank_time(3.5, 1) == 3.5
