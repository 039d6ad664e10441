"""The multi-GPU path of the bench on CPU: two gloo ranks take the maximum of
their step times (the job runs at its slowest replica), and under torchrun
with two ranks the reference arm prints exactly one line, from rank 0.
No GPU is used."""
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
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [0.25, 0.40][rank]
        out[rank] = (bench.max_over_ranks(local_ms, world, "cpu"), bench.whole_job_tokens(16384, world))
    finally:
        dist.destroy_process_group()


def test_gloo_two_ranks_take_the_slowest_step():
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
        res = dict(out)
    assert res[0] == res[1] == (0.40, 32768)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(0.3, 1, "cpu") == 0.3
    assert bench.whole_job_tokens(100, 1) == 100


def test_torchrun_two_ranks_reference_arm_prints_one_line():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--ref-heads", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
