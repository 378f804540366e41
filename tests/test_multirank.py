"""The benchmark's multi-GPU path runs independent replicas (no data-path
collective): each rank times its own steps, the job's step time is the max over
ranks, and whole-job throughput counts every rank's step.  Checked here with two
gloo ranks on the CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local = [3.0, 5.0][rank]
    m = bench.max_over_ranks(local, "cpu")
    out[rank] = (m, bench.job_throughput(m, world))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0][0] == 5.0 and out[1][0] == 5.0
    assert out[0][1] == pytest.approx(2 * 1e3 / 5.0)


def test_single_process_is_identity():
    import bench
    assert bench.max_over_ranks(2.5) == 2.5
    assert bench.job_throughput(2.0, 1) == pytest.approx(500.0)
