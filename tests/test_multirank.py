"""bench.py's multi-rank path on the CPU: two gloo ranks agree on the slowest
rank's time, and under torchrun only rank 0 prints the (single) JSON line.

The product does not shard here (each rank runs an independent replica), so
the only cross-rank steps are the barrier and the max over ranks of the timed
region; these tests run them with world size 2 on the gloo backend.
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


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        elapsed = 1.0 + rank  # rank 1 is the slower one
        got = bench._reduce_max(elapsed, torch.device("cpu"), world)
        dist.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(repr(got))
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    got = [float(open(tmp_path / f"rank{r}.txt").read()) for r in range(2)]
    assert got == [2.0, 2.0]


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench._reduce_max(3.5, torch.device("cpu"), 1) == 3.5


def test_reference_arm_under_torchrun_prints_one_line():
    # two ranks launched as the driver launches them: rank 0 alone times the
    # oracle and prints; the other rank exits 0 without work
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
