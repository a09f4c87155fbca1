"""The N > 1 host logic of bench.py, on CPU with world_size 2 (gloo), no GPU.

The path has no exchange step: every rank runs an independent replica of the workload on its own GPU
(weak scaling), so the only cross-rank operations are the barrier around the timed region and the
maximum of the timings, which rank 0 reports as one whole-job rate.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 0.25 * (rank + 1)], "cpu")
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump(got, f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks(tmp_path):
    """Every rank receives each value's maximum over the ranks (the slowest rank's time)."""
    mp = pytest.importorskip("torch.multiprocessing")
    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world, start_method="spawn")
    for rank in range(world):
        with open(tmp_path / f"rank{rank}.json") as f:
            assert json.load(f) == [2.0, 10.0, 0.5]


def test_max_over_ranks_without_a_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.5], "cpu") == [3.0, 4.5]


def test_job_rate_counts_every_replica():
    """N replicas each doing U units per step at the slowest rank's T ms: N * U / T per ms."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_rate(100.0, 2.0, 1) == pytest.approx(50_000.0)
    assert bench.job_rate(100.0, 2.0, 4) == pytest.approx(200_000.0)
    assert bench.job_rate(1, 4.0, 2) == pytest.approx(500.0)          # steps per second


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    """`bench.py --impl reference` launched as the driver launches N > 1 runs (torchrun, two ranks, on
    this CPU): rank 0 times the oracle and prints one JSON line, the other rank exits 0 silently."""
    pytest.importorskip("torch")
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 1
    assert d["value"] > 0 and d["unit"] == "GB/s" and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
