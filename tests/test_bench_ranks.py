"""The multi-rank parts of bench.py on CPU with the gloo backend, world size 2.

Under torchrun every rank times its own GPU and the job's time is the slowest
rank's; the reference arm (the CPU oracle) runs on rank 0 only and the other
ranks exit 0 without work.  Both are exercised here on the CPU.
"""
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


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    got = bench.max_over_ranks(1.5 + rank, dist, torch.device("cpu"))
    with open(os.path.join(out_dir, f"r{rank}"), "w") as f:
        f.write(repr(got))
    dist.destroy_process_group()


def test_max_over_ranks_gloo(tmp_path):
    mp.start_processes(_worker, args=(2, free_port(), str(tmp_path)), nprocs=2,
                       start_method="spawn")
    assert [float((tmp_path / f"r{r}").read_text()) for r in range(2)] == [2.5, 2.5]


def test_max_over_ranks_single_process():
    import bench
    assert bench.max_over_ranks(3.25, None, torch.device("cpu")) == 3.25


def test_reference_arm_under_torchrun_two_ranks():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node",
           "2", "--master-addr", "127.0.0.1", "--master-port", str(free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--cpu-budget", "0.2"]
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600,
                         env={**os.environ, "OMP_NUM_THREADS": "2"})
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
