"""bench.py's multi-GPU path (replicas, one process per GPU), exercised on the
CPU with the gloo backend at world size 2: the rank reductions the bench uses
for its JSON line (barrier, max of the per-rank time, sum of the per-rank
bytes, whole-job GB/s) and the reference arm's rank handling."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        ranks = bench.RankOps(torch, dist, torch.device("cpu"))
        ranks.barrier()
        local_ms = [3.0, 5.0][rank]          # the slower rank sets the time
        local_bytes = [1e9, 2e9][rank]       # each replica processed its own bytes
        q.put((rank, ranks.max(local_ms), ranks.sum(local_bytes),
               bench.aggregate_gbps(local_bytes, local_ms, ranks)))
        ranks.barrier()
    finally:
        dist.destroy_process_group()


def test_rank_reductions_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    out = sorted(q.get(timeout=10) for _ in range(2))
    for rank, mx, total, gbps in out:
        assert mx == 5.0
        assert total == 3e9
        assert gbps == pytest.approx(3e9 / 5.0 / 1e6)  # GB/s with times in ms


def test_rank_ops_without_a_process_group_return_the_local_value():
    ranks = bench.RankOps(torch, None, torch.device("cpu"))
    ranks.barrier()
    assert ranks.max(2.5) == 2.5 and ranks.sum(7.0) == 7.0
    assert bench.aggregate_gbps(2e9, 4.0, ranks) == pytest.approx(500.0)


def test_reference_arm_prints_only_on_rank_zero():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_line_on_rank_zero():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0", WD_REFERENCE_BUDGET_S="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == bench.UNIT
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and 1 <= cpu["cores"] <= (os.cpu_count() or 1)
    assert cpu["hardware_concurrency"] == os.cpu_count() and cpu["cpu_model"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["value"] > 0
