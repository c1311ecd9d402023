"""The N > 1 path of bench.py on CPU: two gloo ranks.

The decode path has no exchange step, so several GPUs run independent
replicas; what multi-GPU adds is host logic - the slowest rank's time, the
whole-job throughput, and the reference arm running on rank 0 only.  These
tests run that logic as two processes with the gloo backend.
"""
import contextlib
import importlib.util
import io
import json
import os
import socket
import types

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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        r, w, local = b.rank_env()
        assert (r, w, local) == (rank, world, rank)
        dist.barrier()
        local_ms = [3.0, 5.0][rank]          # rank 1 is the slow one
        slowest = b.max_over_ranks(local_ms, w, dist, torch.device("cpu"))
        out[rank] = (slowest, b.job_throughput(w, 1_000_000, slowest))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time_and_job_value():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == out[1]
    slowest, gbs = out[0]
    assert slowest == 5.0
    # two replicas of 1 MB per step in 5 ms
    assert abs(gbs - 2 * 1_000_000 / 5e-3 / 1e9) < 1e-12


def test_single_rank_needs_no_process_group():
    b = _bench()
    assert b.max_over_ranks(7.0, 1) == 7.0
    assert b.job_throughput(1, 10**9, 1000.0) == 1.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    b = _bench()
    args = types.SimpleNamespace(steps=1, warmup=3)
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        b.run_reference(args)
    assert buf.getvalue() == ""                      # other ranks: no work, no line
    monkeypatch.setenv("RANK", "0")
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        b.run_reference(args)
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
