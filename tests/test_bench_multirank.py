"""The multi-rank timing logic of bench.py on CPU: two gloo ranks with
different times agree on the slowest one and on the whole-job throughput."""
import importlib.util
import os
import socket
from pathlib import Path

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parents[1]


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod", ROOT / "bench.py")
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        mine = 10.0 * (rank + 1)  # rank 1 is the slow one
        ms = b.max_over_ranks(mine, world, "cpu")
        out[rank] = (ms, b.job_throughput(1000, world, 5, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    ms, value = res[0]
    assert ms == pytest.approx(20.0)
    # 2 ranks x 1000 units x 5 steps in the slowest rank's 20 ms
    assert value == pytest.approx(2 * 1000 * 5 / 0.020)


def test_single_rank_needs_no_process_group():
    b = _bench()
    assert b.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert b.job_throughput(10, 1, 4, 2.0) == pytest.approx(20000.0)
