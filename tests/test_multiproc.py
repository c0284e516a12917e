"""The benchmark's multi-replica timing path (barrier + max over ranks) with two
gloo ranks on the CPU. The data path has no exchange step, so this is the only
multi-process logic there is."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    dist.barrier()
    t = bench.max_over_ranks(1.5 + rank, dist, "cpu")
    v = bench.job_throughput(100.0, world, t)
    q.put((rank, t, v))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_replicas_report_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert [r[1] for r in res] == [2.5, 2.5]
    assert all(abs(r[2] - 200.0 / 2.5) < 1e-12 for r in res)


def test_single_process_helpers():
    import bench
    assert bench.max_over_ranks(3.0, None, "cpu") == 3.0
    assert bench.job_throughput(10.0, 1, 2.0) == 5.0
