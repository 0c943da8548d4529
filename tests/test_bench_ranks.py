"""The multi-rank bench path on the CPU: two gloo ranks in child processes.

The operator's (sequence, head) pairs are independent, so several GPUs run
replicas: no collective touches the data path, only the timing (a barrier
and the maximum step time over ranks) and the whole-job rate. These tests
run that host logic with world size 2 over gloo on 127.0.0.1."""

import argparse
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        local_ms = 1.5 + rank          # rank 1 is the slow one
        dist.barrier()
        job_ms = bench.max_over_ranks(local_ms, ws, "cpu")
        out[rank] = (job_ms, bench.whole_job_rate(16384, ws, job_ms))
    finally:
        dist.destroy_process_group()


def test_step_time_is_the_maximum_over_two_gloo_ranks():
    ws = 2
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(ws, _free_port(), out), nprocs=ws, join=True)
        res = dict(out)
    assert sorted(res) == [0, 1]
    for rank in range(ws):
        job_ms, rate = res[rank]
        assert job_ms == 2.5                          # every rank sees the slowest rank's time
        assert rate == ws * 16384 / 2.5e-3            # all ranks' tokens over that time


def test_one_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25
    assert bench.whole_job_rate(100, 1, 2.0) == 50000.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = argparse.Namespace(config=1, steps=1, warmup=0)
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(args) is None
    assert buf.getvalue() == ""
