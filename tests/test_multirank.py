"""The replica (N > 1) host path of bench.py on CPU with the gloo backend and two
ranks: the max-over-ranks reduction of the timings, the whole-job figure, and the
reference arm running on rank 0 only (the other ranks return without work)."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 3.5], "cpu")
        out[rank] = got
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_gloo():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == [2.0, 10.0, 3.5] and res[1] == [2.0, 10.0, 3.5]


def test_single_rank_reduction_is_identity_and_aggregate():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.25, 2.5], "cpu") == [1.25, 2.5]
    # 2 replicas x 50 decisions in 600 ms: 6 ms per decision of the job
    assert bench.aggregate_ms_per_decision(600.0, 50, 2) == 6.0


def test_reference_arm_runs_on_rank_zero_only():
    sys.path.insert(0, ROOT)
    import argparse
    import bench
    args = argparse.Namespace(workload="expert_fp8_m50", steps=1, warmup=3)
    assert bench.run_reference(args, rank=1, world=2) is None
