"""Host logic of the multi-GPU benchmark (token-sharded replicas, no
collective on the data path): two gloo ranks on the CPU agree on the slowest
rank's time and on the whole-job throughput."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 10.0 + 5.0 * rank                       # rank 1 is the slower replica
    slowest = bench.max_over_ranks(ms, dist, "cpu")
    value = bench.job_tokens_per_s(64, 100, world, slowest)
    q.put((rank, slowest, value))
    dist.destroy_process_group()


def test_two_gloo_replicas_report_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value in out:
        assert slowest == 15.0
        assert value == pytest.approx(2 * 64 * 100 / 0.015)


def test_single_process_needs_no_collective():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_tokens_per_s(64, 10, 1, 1000.0) == 640.0
