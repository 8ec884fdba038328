"""The benchmark's multi-rank logic on the CPU: two `gloo` ranks.

The decode path shards with no data exchange (replicas: every rank decodes
layers of its own); what N > 1 adds is bench plumbing: the barrier, the
maximum of the ranks' times, rank 0 printing, and disjoint inputs per rank.
"""
import argparse
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(dist, 1.5 + rank, torch.device("cpu"))
        dist.barrier()
        seeds = [bench.layer_seed(rank, li) for li in range(32)]
        out.put((rank, t, seeds))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_disjoint_layers():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    assert [r[1] for r in res] == [2.5, 2.5]           # the max over ranks
    assert not set(res[0][2]) & set(res[1][2])          # each rank its own layers


def test_max_over_ranks_without_a_group_is_the_value():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, 3.25, None) == 3.25


def test_reference_arm_runs_on_rank_zero_only():
    sys.path.insert(0, ROOT)
    import bench
    args = argparse.Namespace(steps=1, warmup=0, gpus=2)
    assert bench.reference_arm(args, 1, 2) is None      # no work, nothing printed
