"""The benchmark's multi-rank logic on CPU: two gloo ranks, max-over-ranks
timing and the whole-job throughput (replicas, no data-path collective)."""

import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(10.0 * (rank + 1), world, "cpu")
    val = bench.job_throughput(world, 4096, 100, ms)
    out.put((rank, ms, val))
    torch.distributed.barrier()
    torch.distributed.destroy_process_group()


def test_two_rank_max_and_throughput():
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [20.0, 20.0]          # the slowest rank's time
    assert all(abs(r[2] - 2 * 4096 * 100 / 0.02) < 1e-6 for r in res)


def test_single_rank_passthrough():
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.job_throughput(1, 10, 2, 1000.0) == 20.0
