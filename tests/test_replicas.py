"""Multi-process path of bench.py on CPU (gloo, world size 2).

Sequences are independent, so N GPUs run N replicas with no exchange; the
only cross-rank logic is the job-level aggregation: units of all ranks over
the slowest rank's time, and rank 0 alone printing.
"""

import importlib.util
import os
import socket

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


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench = _bench()
        # rank r processed 100*(r+1) units in (r+1)*0.5 s
        value, slowest, units = bench.job_throughput(100.0 * (rank + 1), 0.5 * (rank + 1), world)
        q.put((rank, value, slowest, units))
    finally:
        dist.destroy_process_group()


def test_job_throughput_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, value, slowest, units in res:
        assert slowest == pytest.approx(1.0)      # max over ranks
        assert units == pytest.approx(300.0)      # sum over ranks
        assert value == pytest.approx(300.0)      # whole-job units / slowest time


def test_single_rank_is_local():
    bench = _bench()
    assert bench.job_throughput(64.0, 0.002, 1) == (32000.0, 0.002, 64.0)
