"""The multi-rank logic of bench.py on CPU: two gloo ranks on 127.0.0.1.

The layer's path does not shard (replicas only), so the only collective is
the max of the per-rank times; rank 0 alone prints, and the reference arm
runs on rank 0 only.
"""
from __future__ import annotations

import importlib.util
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    b = _bench()
    # rank r measured (10 + r, 20 - r) ms: the job takes the slowest of each
    got = b.max_over_ranks([10.0 + rank, 20.0 - rank], world, "cpu")
    out[rank] = got
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == [11.0, 20.0]
    assert res[1] == [11.0, 20.0]


def test_single_rank_is_identity_and_job_value():
    b = _bench()
    assert b.max_over_ranks([3.5, 7.0], 1, "cpu") == [3.5, 7.0]
    # 2 ranks x 256 tokens x 4 steps in 100 ms -> 20,480 tokens/s
    assert b.job_tokens_per_s(2, 256, 4, 100.0) == pytest.approx(20480.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    b = _bench()
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")

    class Args:
        steps, warmup = 1, 0

    buf = io.StringIO()
    with redirect_stdout(buf):
        b.run_reference(Args(), None)  # no workload needed: rank 1 returns at once
    assert buf.getvalue() == ""
