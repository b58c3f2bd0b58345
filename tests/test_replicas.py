"""Multi-rank plumbing of bench.py on CPU (gloo, world size 2).

The decode path shards by independent (sequence, layer) units with no exchange step, so more GPUs
mean more replicas: the only cross-rank operations are the barrier and the max-over-ranks timing.
These tests run those, and the reference arm under a 2-process launch, without a GPU."""
import json
import os
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dist.barrier()
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, world)      # rank 1 is the slow replica
    out[rank] = (ms, bench.whole_job_rate(world, 64, ms))
    dist.destroy_process_group()


def test_max_over_ranks_gloo():
    world = 2
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, 29511, out), nprocs=world, join=True)
        got = dict(out)
    for rank in range(world):
        ms, rate = got[rank]
        assert ms == 15.0
        assert abs(rate - 2 * 64 / 0.015) < 1e-6


def test_whole_job_rate_single():
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.whole_job_rate(1, 10, 1000.0) == 10.0


def test_reference_arm_two_ranks_prints_one_line():
    """Under a 2-process launch the reference arm (the oracle) runs on rank 0 only; rank 1 exits 0."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", "--master-port=29512", os.path.join(ROOT, "bench.py"), "--impl",
           "reference", "--gpus", "2", "--workload", "tiny_4k", "--steps", "2", "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT,
                       env=dict(os.environ, OMP_NUM_THREADS="1"))
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
