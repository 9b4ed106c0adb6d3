"""The N>1 benchmark path on CPU with two gloo ranks: the timing reduction takes
the slowest rank, whole-job throughput counts every replica, and the reference
arm runs on rank 0 only (the other ranks exit without work)."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    slowest = bench.max_over_ranks(10.0 + 5.0 * rank, torch.device("cpu"))
    value = bench.job_throughput(1e9, slowest, world)

    class Args:
        gpus, steps, warmup = world, 1, 0
    rc = bench.run_reference(Args) if rank == 1 else None
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, slowest, value, rc))


def test_two_gloo_ranks_timing_and_reference_arm():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    out = sorted(q.get(timeout=5) for _ in range(2))
    for rank, slowest, value, rc in out:
        assert slowest == 15.0                      # the slowest rank's time
        assert value == pytest.approx(2 * 1e9 / 0.015 / 1e9)
    assert out[1][3] == 0                            # rank 1: reference arm exits without work


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, torch.device("cpu")) == 3.5
    assert bench.job_throughput(2e9, 1000.0, 1) == pytest.approx(2.0)
