"""The multi-rank plumbing of bench.py (replicas: one process per GPU, no data-path collective)
on CPU with the gloo backend and two ranks: rendezvous from the environment, the barrier
around the timed region, the max over ranks of the timed total, and the reference arm printing
on rank 0 only."""
import os
import socket
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update({"WORLD_SIZE": str(world), "RANK": str(rank), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch.distributed as dist
    import bench
    w, r, local = bench.dist_setup(None)
    bench.barrier(w)
    # each rank times a different total; the job's time is the slowest rank's
    m = bench.max_over_ranks(10.0 + 5.0 * r, w)
    bench.barrier(w)
    q.put((r, w, local, dist.get_backend(), m))
    dist.destroy_process_group()


def test_two_rank_rendezvous_barrier_and_max():
    import torch
    import torch.multiprocessing as tmp
    if torch.cuda.is_available():
        pytest.skip("this test covers the CPU (gloo) path")
    ctx = tmp.get_context("spawn")
    q = ctx.SimpleQueue()
    world, port = 2, _free_port()
    tmp.start_processes(_rank_main, args=(world, port, q), nprocs=world, start_method="spawn")
    got = sorted(q.get() for _ in range(world))
    assert [g[0] for g in got] == [0, 1]
    for r, w, local, backend, m in got:
        assert w == world and local == r and backend == "gloo"
        assert m == 15.0  # max over ranks of 10 and 15


def test_reference_arm_prints_on_rank_zero_only(capsys, monkeypatch):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    class A:  # the fields run_reference reads before it returns on a non-zero rank
        M, seed, steps, warmup = 32, 0, 1, 0
    bench.run_reference(A())
    assert capsys.readouterr().out == ""
