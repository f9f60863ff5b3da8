"""The benchmark's multi-rank aggregation (replicas: one independent batch per
rank, no collective on the data path) on two CPU ranks over gloo: the step
time is the slowest rank's, the throughput counts every rank's batch, and
the reference arm prints from rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [0.25, 0.40][rank]                  # rank 1 is the slower one
        ms = bench.max_over_ranks(local_ms, world, "cpu")
        value = bench.job_tflops(7.4e9, world, ms)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"ms": ms, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn")
    r = [json.load(open(tmp_path / f"rank{i}.json")) for i in range(2)]
    assert r[0]["ms"] == r[1]["ms"] == pytest.approx(0.40)
    assert r[0]["value"] == pytest.approx(2 * 7.4e9 / 0.40e-3 / 1e12)


def test_single_rank_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.5, 1) == 1.5
    assert bench.job_tflops(1e12, 1, 1000.0) == pytest.approx(1.0)


def test_reference_arm_prints_on_rank0_only():
    """Two ranks of the reference arm (oracle on the host, tiny workload): one
    JSON line from rank 0, rank 1 exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--gpus", "2", "--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT,
                         env={**os.environ, "OMP_NUM_THREADS": "1"})
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0


def test_gpus_flag_must_match_world_size():
    """--gpus N without N ranks is refused (exit code non-zero) instead of
    silently measuring one GPU."""
    env = {**os.environ, "WORLD_SIZE": "1", "RANK": "0"}
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--impl", "reference",
                          "--workload", "tiny", "--steps", "1"], capture_output=True, text=True, timeout=300,
                         cwd=ROOT, env=env)
    assert out.returncode != 0 and "WORLD_SIZE" in out.stderr
