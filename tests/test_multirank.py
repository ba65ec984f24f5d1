"""The multi-rank host logic of bench.py, on CPU with gloo (world size 2).

Under torchrun every rank runs an independent copy of the workload; the only
cross-rank traffic is a barrier around the timed region and the max over ranks
of the timed total.  These tests run that logic on two gloo ranks, and check
that the reference arm leaves all work to rank 0.
"""
import io
import os
import socket
import sys
import types
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        bench.barrier(ws)
        # each rank's "timed total"; the job's time is the slowest rank's
        got = bench.max_over_ranks(1.5 + rank, ws, torch.device("cpu"))
        bench.barrier(ws)
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_barrier_and_max_over_ranks_gloo():
    ws = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(ws, _free_port(), out), nprocs=ws, start_method="spawn", join=True)
        assert dict(out) == {0: 1.5 + ws - 1, 1: 1.5 + ws - 1}


def test_single_rank_needs_no_process_group():
    import bench

    assert bench.max_over_ranks(3.25, 1, torch.device("cpu")) == 3.25
    bench.barrier(1)  # no process group: must not touch torch.distributed


def test_reference_arm_runs_on_rank_zero_only():
    import bench

    args = types.SimpleNamespace(workload="prefill_h16_t8k", warmup=3, steps=1, gpus=2)
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.run_reference(args, ws=2, rank=1)
    assert buf.getvalue() == ""


@pytest.mark.parametrize("env,expect", [({}, (1, 0, 0)), ({"WORLD_SIZE": "2", "RANK": "1", "LOCAL_RANK": "1"}, (2, 1, 1))])
def test_dist_env(monkeypatch, env, expect):
    import bench

    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    for k, v in env.items():
        monkeypatch.setenv(k, v)
    assert bench.dist_env() == expect
