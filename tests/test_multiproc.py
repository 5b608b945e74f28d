"""The multi-process (torchrun) paths of bench.py on CPU: two gloo ranks.

Every workload shards by batch with no data-path collective (weak scaling:
each rank runs its own full workload); the only cross-rank step is the
timing, a max over ranks.  These tests cover that host logic and the
reference arm's rank handling without a GPU."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(10.0 + 5.0 * rank, world)   # rank 1 is slower
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_gloo():
    import torch.multiprocessing as tmp
    ctx = tmp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res == {0: 15.0, 1: 15.0}


def test_whole_job_value_is_weak_scaling():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.whole_job_value(2 ** 30, 1, 1.0)
    assert abs(bench.whole_job_value(2 ** 30, 4, 1.0) - 4 * one) < 1e-6
    assert abs(one - 2 ** 30 / 1e-3 / 1e9) < 1e-6


def test_reference_arm_under_torchrun_prints_once():
    # Rank 0 alone runs the CPU oracle and prints one JSON line; rank 1 exits
    # 0 without work.
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(30500 + os.getpid() % 1000),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "0", "--ref-step-seconds", "0.3", "--config", "c1"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


def test_planned_passes_follow_the_planner():
    # The HBM pass count bench.py assumes before a plan exists mirrors the
    # planner's own rule: factors of at most 9 bits, at least two passes.
    import bench
    assert bench.planned_passes(26, 9) == 3
    assert bench.planned_passes(15, 9) == 2
    assert bench.planned_passes(30, 9) == 4
    assert bench.planned_passes(18, 13) == 2
