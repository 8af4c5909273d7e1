"""Two gloo ranks on the CPU: the bench's multi-GPU aggregation (replicas only:
every rank runs the sweep on its own GPU; the job's time is the slowest rank's
and its throughput counts every rank's work)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    import bench

    ms = bench.slowest_rank_ms(1.0 + 2.0 * rank, world, "cpu")
    q.put((rank, ms, bench.job_tflops(1.0e12, world, ms)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert sorted(r for r, _, _ in got) == [0, 1]
    for _, ms, tf in got:
        assert ms == 3.0  # rank 1's 3 ms, seen by both ranks
        assert tf == pytest.approx(1.0e12 * 2 / 3.0e-3 / 1e12)


def test_one_rank_is_unchanged():
    import bench

    assert bench.slowest_rank_ms(1.5, 1, "cpu") == 1.5
    assert bench.job_tflops(2.0e12, 1, 2.0) == pytest.approx(1000.0)
