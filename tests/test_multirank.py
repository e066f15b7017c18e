"""The N > 1 host path of the benchmark, on CPU with the gloo backend.

Every rank runs its own replica of the batch (the data path has no
collective); the job's time is the slowest rank's, and its throughput counts
the bytes of every replica.  These tests run two gloo ranks on 127.0.0.1:
the max-over-ranks reduction the benchmark uses, the throughput formula, and
the reference arm launched by torchrun with two processes (rank 0 alone
prints one line, the other exits 0 without work).
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, values, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.max_over_ranks(values[rank])
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_gloo():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    values = [12.5, 40.25]
    mp.start_processes(_worker, args=(world, port, values, out), nprocs=world, join=True,
                       start_method="spawn")
    assert out[0] == out[1] == 40.25


def test_max_over_ranks_without_group_is_identity():
    assert bench.max_over_ranks(3.5) == 3.5


def test_job_throughput_counts_every_replica():
    # 2 replicas x 10 steps x 1 GB in 5 ms -> 4000 GB/s
    assert bench.job_throughput(10 ** 9, 10, 2, 5.0) == pytest.approx(4000.0)
    assert bench.job_throughput(10 ** 9, 10, 1, 5.0) == pytest.approx(2000.0)


def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--workload", "tiny", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--ref-rows", "2"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2
    assert rec["value"] > 0 and rec["cpu_baseline"]["kind"] == "oracle"
    assert rec["e2e"]["h2d_bytes_per_step"] == 0


def test_gpus_flag_without_a_launcher_starts_that_many_ranks():
    """`bench.py --gpus 2` run directly (the form the scaling run uses
    without torchrun) relaunches itself under torch.distributed.run with two
    processes; the reference arm's single line then reports both ranks."""
    cmd = [sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--gpus", "2",
           "--steps", "1", "--warmup", "3", "--ref-rows", "2"]
    env = {k: v for k, v in os.environ.items()
           if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2
