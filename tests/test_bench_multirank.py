"""The benchmark's multi-rank logic on CPU: two gloo ranks (torchrun-style
environment), the slowest rank's time taken for the job, the whole-job rate
summed over replicas, and the reference arm's non-zero ranks exiting without
work."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        class A:
            gpus = world
        w, r, l = bench.dist_setup(A)
        elapsed = 10.0 + 5.0 * rank  # rank 1 is the slower one
        job = bench.max_over_ranks(elapsed, "cpu")
        rate = bench.whole_job_rate(1e9, 4, job, w)
        q.put((r, w, l, job, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for r, (rank, world, local, job, rate) in enumerate(res):
        assert (rank, world, local) == (r, 2, r)
        assert job == 15.0                        # max over ranks
        assert rate == pytest.approx(2 * 1e9 * 4 / 15e-3 / 1e9)


def test_single_process_is_its_own_max():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.whole_job_rate(2e9, 10, 1000.0, 1) == pytest.approx(20.0)


def test_reference_arm_nonzero_rank_exits_without_work(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        gpus = 2
        config = "lookup16"
        steps = 1
        warmup = 0
    assert bench.run_reference(A) == 0
