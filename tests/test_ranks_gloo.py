"""Multi-process host logic of bench.py's replica runs (one process per GPU,
launched by torchrun), on the CPU with the gloo backend and world size 2:
the timing reduction takes the slowest rank, and the whole-job throughput
counts every rank's tokens against that time. No GPU is used."""
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


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        ms = [12.5, 20.0][rank]  # rank 1 is the slow one
        dist.barrier()
        slowest = b.max_over_ranks(ms, world, torch.device("cpu"))
        tok = b.job_tokens_per_s(8192, 10, world, slowest)
        out[rank] = (slowest, tok)
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_reduction():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world,
                           start_method="spawn", join=True)
        res = dict(out)
    for rank in range(world):
        slowest, tok = res[rank]
        assert slowest == 20.0
        assert tok == pytest.approx(2 * 8192 * 10 / 0.020)


def test_single_rank_is_identity():
    b = _bench()
    assert b.max_over_ranks(3.25, 1, torch.device("cpu")) == 3.25
    assert b.job_tokens_per_s(100, 4, 1, 2.0) == pytest.approx(200000.0)
