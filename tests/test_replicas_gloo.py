"""bench.py across ranks, on the CPU: two processes joined by the gloo
backend stand in for two GPUs running independent replicas of the workload.

The whole job's time is the slowest rank's, and its throughput counts the
units of every replica; the reference arm runs on rank 0 only.
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


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_setup(None)
        ms = 10.0 * (rank + 1)          # rank 1 is the slower replica
        slow = bench.slowest_rank_ms(ms, dist, "cpu")
        value = bench.job_throughput(w, 4, 1000, slow)
        q.put((rank, w, r, local, slow, value))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_slowest_rank_time_and_job_throughput():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        results = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(60)
    assert [p.exitcode for p in procs] == [0, 0]
    for rank, w, r, local, slow, value in results:
        assert (w, r, local) == (2, rank, rank)
        assert slow == 20.0                                  # max over the ranks
        assert value == pytest.approx(2 * 4 * 1000 / 0.020)  # both replicas' units


def test_one_rank_is_its_own_job():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank_ms(12.5, None, "cpu") == 12.5
    assert bench.job_throughput(1, 10, 8192, 5.0) == pytest.approx(10 * 8192 / 0.005)


def test_reference_arm_runs_on_rank_zero_only(capsys):
    sys.path.insert(0, ROOT)
    import bench
    from learned_group_sparse_gb300 import synth
    # a rank other than 0 returns at once: no device, no oracle, no output
    assert bench.run_reference(None, synth.workload(1), 2, 1) is None
    assert capsys.readouterr().out == ""
