"""The bench's multi-GPU path is replicas only: each rank runs the whole decode on its
own GPU, and rank 0 reports the units of all ranks over the slowest rank's time.  The
host-side pieces run here as world-size-2 gloo process groups on the CPU."""
import os
import socket

import pytest

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, seconds, out):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    slowest = bench.max_over_ranks(seconds[rank], "cpu")
    out[rank] = (slowest, bench.job_throughput(1000.0, world, slowest))
    dist.barrier()
    dist.destroy_process_group()


def test_slowest_rank_sets_the_job_throughput():
    import torch.multiprocessing as mp
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(2, port, [1.5, 2.5], out), nprocs=2, join=True)
        res = dict(out)
    # both ranks see the slowest time; the job did 2 x 1000 units in 2.5 s
    assert res[0] == res[1] == (2.5, 800.0)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.job_throughput(10.0, 1, 2.0) == 5.0


def test_reference_arm_runs_on_rank_0_only(capsys, monkeypatch):
    # other ranks exit without work and print nothing
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    args = bench_args(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert bench.reference_arm(args) is None
    assert capsys.readouterr().out == ""


def bench_args(argv):
    import argparse
    ap = argparse.ArgumentParser()
    ap.add_argument("--impl")
    ap.add_argument("--steps", type=int)
    ap.add_argument("--warmup", type=int)
    ap.add_argument("--workload", default=bench.WORKLOAD)
    ap.add_argument("--ref-seconds", type=float, default=1.0)
    return ap.parse_args(argv)
