"""The multi-rank bench path on CPU: two gloo ranks (no GPU).

bench.py runs one independent replica of the workload per GPU ("replicas
only": all N simulated ranks of the method live in one GPU's HBM).  What
crosses ranks is the timing: the slowest rank's time, and the whole-job
throughput of all ranks' units.  These run here as two processes.
"""

import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank                  # rank 1 is the slow one
        slowest = bench.max_over_ranks(local_ms, dist, "cpu")
        value = bench.job_throughput(1_000_000, dist.get_world_size(), slowest * 1e-3)
        dist.barrier()
        q.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_units():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slowest, value in got:
        assert slowest == 15.0
        assert value == pytest.approx(2 * 1_000_000 / 0.015)


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_throughput(10, 1, 2.0) == 5.0


def test_reference_arm_other_ranks_exit_quietly(capsys, monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.main(["--impl", "reference", "--gpus", "2", "--steps", "3", "--warmup", "3"]) == 0
    assert capsys.readouterr().out == ""
