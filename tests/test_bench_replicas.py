"""The multi-GPU path of bench.py is independent replicas: every timed quantity is the maximum
over ranks and whole-job throughput counts all ranks' tokens.  Checked here with two gloo
ranks on the CPU (no GPU, no NCCL)."""
import importlib.util
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench = _bench()
        local = {"decode_s": 1.0 + rank, "prefill_s": 0.5 - 0.25 * rank, "total_ms": 100.0 * (rank + 1)}
        q.put((rank, bench.aggregate_replicas(local, world, torch.device("cpu"))))
    finally:
        dist.destroy_process_group()


def test_replica_times_are_the_max_over_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    expect = {"decode_s": 2.0, "prefill_s": 0.5, "total_ms": 200.0}
    assert got[0] == expect and got[1] == expect
    # whole-job throughput as bench.py forms it: all ranks' tokens over the slowest rank's time
    tokens_per_rank = 64 * 512
    assert world * tokens_per_rank / got[0]["decode_s"] == pytest.approx(32768.0)


def test_single_process_passes_times_through():
    bench = _bench()
    local = {"decode_s": 1.5, "prefill_s": 0.2, "total_ms": 7.0}
    assert bench.aggregate_replicas(local, 1, torch.device("cpu")) == local


def test_reference_arm_runs_on_rank_zero_only(capsys):
    bench = _bench()

    class Args:
        gpus, steps, warmup = 2, 1, 0

    bench.run_reference(Args, rank=1)  # the other ranks exit without work
    assert capsys.readouterr().out == ""
