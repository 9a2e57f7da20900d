"""Host-side pieces of the benchmark: whole-job throughput over replicas, the
max-over-ranks timing on a real 2-rank process group (gloo, CPU), and the
reference arm's rank handling.  No GPU needed."""
import os
import socket
import sys
from pathlib import Path

import pytest
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parent.parent
sys.path.insert(0, str(ROOT))
import bench  # noqa: E402


def test_job_throughput_counts_every_replica():
    flops = 2.0 * 8192 ** 3
    one = bench.job_throughput(flops, 10, 1, 7.0)
    assert abs(one - flops * 10 / 7e-3 / 1e12) < 1e-9
    # four replicas doing the same work in the same (slowest) time: four times the throughput
    assert abs(bench.job_throughput(flops, 10, 4, 7.0) - 4 * one) < 1e-9


def test_max_over_ranks_without_process_group():
    assert bench.max_over_ranks(3.5) == 3.5


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 5.0 + 2.0 * rank              # rank 1 is the slow one
        m = bench.max_over_ranks(local_ms)
        q.put((rank, m, bench.job_throughput(1e12, 3, world, m)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, tput in got:
        assert m == 7.0                           # both ranks see the slowest rank's time
        assert abs(tput - 2 * 1e12 * 3 / 7e-3 / 1e12) < 1e-9


def test_reference_arm_non_zero_rank_does_nothing(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        workload, steps, warmup, cpu_seconds = "square8192_bf16", 1, 3, 1.0

    assert bench.run_reference(Args()) is None
