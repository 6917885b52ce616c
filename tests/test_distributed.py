"""Multi-process host logic of the benchmark on CPU (gloo, world size 2).

The decode path does not shard with an exchange step: N GPUs run N
independent replicas, so the only cross-rank logic is the timing reduction
(the slowest rank's time, whole-job throughput) and the reference arm's
"rank 0 alone" rule. Both run here on CPU ranks.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        elapsed = [40.0, 55.5][rank]  # rank 1 is the slow one
        m = bench.max_over_ranks(elapsed, "cpu", world)
        v = bench.whole_job_gbs(1_000_000, 10, m, world)
        results[rank] = (m, v)
    finally:
        dist.destroy_process_group()


def test_timing_reduction_takes_the_slowest_rank():
    import torch.multiprocessing as mp

    mgr = mp.Manager()
    results = mgr.dict()
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, results), nprocs=2, start_method="spawn")
    assert results[0] == results[1]
    m, v = results[0]
    assert m == 55.5
    # two replicas of 1 MB steps, 10 steps in the slowest rank's 55.5 ms
    assert v == pytest.approx(2 * 1_000_000 * 10 / 55.5e-3 / 1e9)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(12.5, "cpu", 1) == 12.5
    assert bench.whole_job_gbs(2_000_000, 5, 10.0, 1) == pytest.approx(1.0)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    """`bench.py --impl reference` launched as the driver launches N > 1:
    rank 0 times the oracle and prints one JSON line, rank 1 exits 0 without
    work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle"
