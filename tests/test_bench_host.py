"""Host-side logic of bench.py on CPU: the multi-rank reduction (gloo,
world size 2) and the whole-job aggregate, plus the reference arm's
bookkeeping on a tiny layer."""
import json
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [0.25, 0.40][rank]
        ms_max = bench.max_over_ranks(ms, world)
        val = bench.aggregate_gbs(1_000_000_000, world, ms_max)
        out[rank] = (ms_max, val)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = 29500 + os.getpid() % 1000
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, start_method="spawn")
    for r in range(2):
        ms_max, val = out[r]
        assert ms_max == pytest.approx(0.40)
        # two replicas of 1 GB each in 0.40 ms
        assert val == pytest.approx(2e9 / 0.40e-3 / 1e9)


def test_single_rank_aggregate():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.5, 1) == 0.5
    assert bench.aggregate_gbs(1315927040, 1, 0.5) == pytest.approx(2631.85408)


def test_reference_arm_prints_one_line():
    # the oracle as the reference arm, on a one-layer-sized workload
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "1"], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0
