"""The N > 1 path of bench.py on CPU: two ranks over gloo.

Every GPU replica runs the same step on its own data; the only exchange is
the timing, reduced to the slowest rank before the whole-job throughput is
formed. This checks that reduction and the throughput formula with two
processes, and that the reference arm leaves ranks other than 0 idle."""

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took (10 + r) ms for the steps, (20 - r) ms end to end
        got = bench.max_over_ranks([10.0 + rank, 20.0 - rank, 1.5], "cpu")
        value = bench.job_throughput(world, 32768, 50, got[0])
        ws, r, local = bench._dist()
        q.put((rank, got, value, (ws, r, local)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, value, env in results:
        assert got == [11.0, 20.0, 1.5]  # element-wise max over the two ranks
        assert value == pytest.approx(2 * 32768 * 50 / 0.011)
        assert env == (world, rank, rank)


def test_one_rank_is_the_identity():
    assert bench.max_over_ranks([3.0, 4.0], "cpu") == [3.0, 4.0]
    assert bench.job_throughput(1, 100, 10, 1000.0) == pytest.approx(1000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")

    class Args:
        steps, warmup = 1, 0

    assert bench.run_reference(Args()) is None  # no oracle work on rank 1
