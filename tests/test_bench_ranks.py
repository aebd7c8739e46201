"""The multi-rank path of bench.py, on the CPU.

Under torchrun every rank runs one independent replica of the decode step on its own GPU
(the path partitions by agent; no collective on the data path).  The job's step time is its
slowest rank's, and its throughput is the sum over replicas.  Here two `gloo` ranks (one
process each, as torchrun starts them) run the same reductions bench.py uses, and the
reference arm is launched as rank 1 and rank 0 of a two-rank job.
"""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, step_ms: list, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(step_ms[rank])
        q.put((rank, slowest, bench.job_tokens_per_s(world, 8, 32, slowest / 1000)))
    finally:
        dist.destroy_process_group()


def test_one_rank_keeps_its_own_time():
    assert bench.max_over_ranks(3.25) == 3.25
    # 8 agents x 32 layers per 1.6 ms step
    assert bench.job_tokens_per_s(1, 8, 32, 1.6e-3) == pytest.approx(160000.0)


def test_two_gloo_ranks_take_the_slowest_replica_and_sum_the_tokens():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    step_ms = [1.5, 1.75]  # rank 1 is the slower replica
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, step_ms, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        results = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    for rank, slowest, value in results:
        assert slowest == 1.75
        assert value == pytest.approx(2 * 8 * 32 / 1.75e-3)


def _reference_run(rank: int, world: int):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--config", "tiny_decode", "--steps", "1", "--warmup", "3"],
                          capture_output=True, text=True, env=env, timeout=300)


def test_reference_arm_prints_from_rank_zero_only():
    other = _reference_run(1, 2)
    assert other.returncode == 0, other.stderr
    assert other.stdout.strip() == ""
    first = _reference_run(0, 2)
    assert first.returncode == 0, first.stderr
    lines = [ln for ln in first.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "tokens/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_percentiles_are_nearest_rank():
    xs = [5.0, 1.0, 4.0, 2.0, 3.0, 9.0, 8.0, 7.0, 6.0, 10.0]
    assert bench.percentiles(xs) == {"p10": 1.0, "p50": 5.0, "p90": 9.0}
    assert bench.percentiles([2.5]) == {"p10": 2.5, "p50": 2.5, "p90": 2.5}
