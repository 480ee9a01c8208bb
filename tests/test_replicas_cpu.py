"""Multi-GPU runs are replicas only: every rank runs the whole path on its
own scene and the benchmark reduces (slowest time, total voxels) after the
timed region.  This checks that host logic with two gloo ranks on the CPU,
and that the reference arm does its work on rank 0 alone."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r timed 1 + r seconds over 100 * (r + 1) voxels
        t, n = bench.reduce_over_ranks(1.0 + rank, 100 * (rank + 1), "cpu", world)
        w, s = bench.make_workload(0, rank)
        q.put((rank, t, n, s.coords[:, 1:3].tobytes(), s.n))
    finally:
        dist.destroy_process_group()


def test_two_replicas_reduce_max_time_and_total_units():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, n, _, _ in res:
        assert t == 2.0  # the slowest rank's time
        assert n == 300.0  # voxels of both replicas
    # each replica draws its own scene of the same recipe and size
    assert res[0][3] != res[1][3]
    assert res[0][4] == res[1][4] == 200


def test_single_rank_reduction_is_the_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(0.5, 1234, "cpu", 1) == (0.5, 1234.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"])
    bench.main()
    assert capsys.readouterr().out == ""
