"""The multi-rank (N > 1) host logic of bench.py on CPU with the gloo
backend: two ranks, each a replica with its own batch.  No GPU is needed:
the timing reduction and the whole-job rate are plain host code, and the
reference arm (the oracle on host cores) runs on rank 0 only."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, ws, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        local_ms = [80.0, 95.5][rank]                   # rank 1 is the slower replica
        worst = bench.max_over_ranks(local_ms, ws)
        rate = bench.whole_job_rate(208_896_000, ws, worst / 1000.0)
        q.put((rank, worst, rate))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_takes_the_slowest_rank_and_sums_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, worst, rate in got:
        assert worst == 95.5
        # both replicas' bytes over the slowest replica's time
        assert abs(rate - 2 * 208_896_000 / 95.5e-6 / 1e9) < 1e-6 * rate


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5, 1) == 12.5
    assert abs(bench.whole_job_rate(1_000_000_000, 1, 1000.0) - 1.0) < 1e-12


def test_reference_arm_under_torchrun_prints_one_line_from_rank_zero():
    env = dict(os.environ, PYTHONPATH=ROOT)
    r = subprocess.run(
        [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
         "--master-addr", "127.0.0.1", "--master-port", str(29700 + os.getpid() % 200),
         os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
         "--warmup", "0", "--workload", "tiny_f32", "--cpu-sample-seconds", "0.5"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
