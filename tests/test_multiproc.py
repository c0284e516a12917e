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


def test_clock_sampler_without_a_gpu_reports_instead_of_failing():
    # no GPU and no NVML here: the sampler falls back to nvidia-smi and, without it, returns
    # an empty record naming why, and a window that holds no sample is not an error
    import torch

    import bench
    c = bench.clock_sampler(0)
    c.start()
    out = c.stop((0.0, 1.0))
    assert set(out) >= {"sm_mhz", "sm_max_mhz", "reasons", "samples"}
    if not torch.cuda.is_available():
        assert out["samples"] == 0 and out["sm_mhz"] is None


def test_nvml_window_selects_the_samples_inside_it():
    # the NVML sampler's reduction, on hand-made samples: (host time, SM MHz, W, reasons)
    import bench
    s = bench.NvmlClocks.__new__(bench.NvmlClocks)
    s.max_mhz, s.stop_flag = 2070.0, False
    s.thread = type("T", (), {"join": lambda self, timeout=None: None})()
    s.samples = [(0.5, 1500.0, 100.0, 0x0), (1.0, 2070.0, 300.0, 0x4), (1.5, 2060.0, 310.0, 0x0),
                 (2.0, 2070.0, 305.0, 0x0), (3.0, 900.0, 90.0, 0x40)]
    out = s.stop((0.9, 2.1))
    assert out["samples"] == 3 and out["scope"] == "timed loop"
    assert out["sm_mhz"] == 2070.0 and out["reasons"] == ["sw_power_cap"]
    assert out["power_w_max"] == 310.0
    s.stop_flag = False
    out = s.stop((5.0, 6.0))  # nothing inside: every sample, said so
    assert out["samples"] == 5 and out["scope"] == "whole run"
    assert out["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
