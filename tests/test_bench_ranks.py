"""bench.py's multi-rank host logic on CPU ranks (gloo, world size 2).

Every rank times its own replica; the job's time is the slowest rank's and the
job's throughput counts every rank's units over that time.  No GPU: the ranks
exchange float64 tensors on the CPU.
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


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        b.barrier(world)
        job_ms = b.max_over_ranks(times[rank], world, torch.device("cpu"))
        out[rank] = (job_ms, b.job_rate(world, 1000.0, job_ms))
        b.barrier(world)
    finally:
        dist.destroy_process_group()


def test_job_time_is_the_slowest_rank():
    world, port = 2, _free_port()
    times = [12.5, 20.0]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, times, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        job_ms, rate = res[r]
        assert job_ms == 20.0                       # every rank agrees on the max
        assert rate == pytest.approx(2 * 1000.0 / 0.020)


def test_single_process_helpers_need_no_process_group():
    b = _bench()
    b.barrier(1)
    assert b.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5
    assert b.job_rate(1, 10.0, 100.0) == pytest.approx(100.0)


def test_source_hash_ignores_comments_but_not_code(tmp_path):
    b = _bench()
    a = tmp_path / "a.cu"
    c = tmp_path / "c.cu"
    d = tmp_path / "d.cu"
    a.write_text("// header\nint f(int x) { return x + 1; }  /* tail */\n")
    c.write_text("// another header\n\nint f(int x) {\n  return x + 1;  // same code\n}\n")
    d.write_text("int f(int x) { return x + 2; }\n")
    assert b.src_hash([str(a)]) == b.src_hash([str(c)])
    assert b.src_hash([str(a)]) != b.src_hash([str(d)])
