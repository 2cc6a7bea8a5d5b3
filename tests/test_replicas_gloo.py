"""The multi-GPU path of bench.py is replicas only (every rank runs the same
workload on its own GPU; no data-path collective). Its host logic -- the
max-over-ranks of the timed region, the barrier, and rank 0 alone printing the
reference arm -- is checked here with two gloo ranks on the CPU."""
import io
import json
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank "measured" a different duration; all must see the slowest
        v = bench.reduce_max(10.0 + rank * 2.5, world, torch.device("cpu"))
        bench.barrier(world)
        results[rank] = v
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        results = m.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        assert dict(results) == {0: 12.5, 1: 12.5}


def test_reference_arm_prints_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        steps, warmup = 1, 0

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.reference_arm(Args())
    assert buf.getvalue() == ""
    monkeypatch.setenv("RANK", "0")
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.reference_arm(Args())
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
