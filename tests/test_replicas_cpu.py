"""Multi-GPU bookkeeping of bench.py, run as two gloo ranks on the CPU.

Every pair is independent and each GPU holds its own pool replica, so the
multi-GPU bench runs replicas with no collective on the data path.  The only
cross-rank steps are the barrier around the timed region and the max of the
ranks' times; the whole-job value counts every rank's bytes over that max.
"""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

REPO = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, REPO)
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        local_ms = [120.0, 150.0][rank]
        bench.barrier(world)
        slowest = bench.max_over_ranks(local_ms, world)
        value = bench.aggregate_gbs(world, 10, 4 * 2 ** 30, slowest)
        out[rank] = (slowest, value)
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_count_all_bytes():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                           start_method="spawn", join=True)
        got = dict(out)
    assert got[0][0] == got[1][0] == 150.0
    want = 2 * 10 * 4 * 2 ** 30 / 0.150 / 1e9
    assert abs(got[0][1] - want) < 1e-6 and got[0][1] == got[1][1]


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, REPO)
    import bench

    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert abs(bench.aggregate_gbs(1, 2, 1e9, 1000.0) - 2.0) < 1e-12


def test_cpu_list_parsing_for_host_placement():
    """The bench binds pool allocation to the CPUs sysfs lists as local to the GPU."""
    import bench
    assert bench._cpulist("0-3,8,10-11") == {0, 1, 2, 3, 8, 10, 11}
    assert bench._cpulist("") == set() and bench._cpulist(None) == set()
    assert bench._cpulist("5") == {5}
