"""The bench's multi-rank plumbing on CPU with gloo (world size 2): the max-over-ranks
step time, and the reference arm under torchrun (rank 0 prints the one JSON line, the
other rank exits 0 without work)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench

    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.max_over_ranks(1.5 + rank, "cpu")
    finally:
        torch.distributed.destroy_process_group()


@pytest.mark.timeout(300)
def test_max_over_ranks_gloo_world2():
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank_main, args=(2, _free_port(), out), nprocs=2, join=True, start_method="spawn")
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_max_over_ranks_single_process_is_identity():
    import bench

    assert bench.max_over_ranks(3.25, "cpu") == 3.25


@pytest.mark.timeout(600)
def test_reference_arm_under_torchrun_world2():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference", "--workload",
           "contig4096", "--steps", "1", "--gpus", "2"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
