"""The bench's multi-rank reduction on two gloo ranks (CPU): every rank
reports its own time, the job takes the slowest, and the whole-job rate
counts every replica's work.  The path on the GPUs is the same code on NCCL
(one replica per GPU, no collective on the data path)."""
import importlib.util
import multiprocessing as mp
import os
import socket

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def rank_main(rank, world, port, times, out):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = load_bench()
        t = b.max_over_ranks(times[rank], world, torch.device("cpu"))
        out.put((rank, t, b.whole_job_rate(1e12, world, t)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    times = [12.5, 20.0]
    port = free_port()
    procs = [ctx.Process(target=rank_main, args=(r, 2, port, times, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, rate in got:
        assert t == 20.0
        # 2 replicas x 1 TFLOP in 20 ms
        assert rate == pytest.approx(100.0)


def test_one_rank_needs_no_process_group():
    b = load_bench()
    assert b.max_over_ranks(3.0, 1, None) == 3.0
    assert b.whole_job_rate(2e12, 1, 10.0) == pytest.approx(200.0)


def test_every_workload_has_an_oracle_case():
    """The reference arm and the CPU baseline time the oracle on a case of
    each workload the bench offers."""
    b = load_bench()
    assert set(b.ORACLE_SPECS) == set(b.WORKLOADS)
