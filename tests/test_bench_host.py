"""Host-side checks of bench.py (no GPU): the multi-rank aggregation over gloo with
world size 2, the algorithmic byte count, and the reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, elapsed, queue):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        worst = bench.max_over_ranks(elapsed[rank], dist, "cpu")
        value = bench.replica_gbs(world, 10**9, 4, worst)
        queue.put((rank, worst, value))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_and_sum_the_bytes():
    world, port = 2, _free_port()
    elapsed = [8.0, 12.5]  # ms per rank for 4 steps of 1 GB each
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, elapsed, queue))
             for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(queue.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, worst, value in results:
        assert worst == 12.5
        assert value == pytest.approx(2 * 4 * 1e9 / 12.5e-3 / 1e9)


def test_single_process_aggregation_is_identity():
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.replica_gbs(1, 2 * 10**9, 10, 1000.0) == pytest.approx(20.0)


def test_step_bytes_count_each_listed_row_once():
    wl = workloads.prefix_shared_workload([100], [5, 7], 2, n_qo_heads=32, n_kv_heads=8,
                                          head_dim=128, layers=3, seed=1)
    nb = bench.step_bytes(wl)
    unique = 100 + 5 + 7
    logical = 2 * 100 + 5 + 7
    row = 8 * 128 * 2
    per_q = 2 * 32 * 128 * 2 * 2 + 2 * 32 * 4  # q + out + lse for 2 requests
    idx = logical * 4 + 3 * 4
    assert nb["attn_per_layer"] == unique * 2 * row + idx + per_q
    assert nb["attn_logical_per_layer"] == logical * 2 * row + idx + per_q
    assert nb["append_per_layer"] == 2 * (2 * row * 2) + 2 * 4
    assert nb["step"] == 3 * (nb["attn_per_layer"] + nb["append_per_layer"])


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "1", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
