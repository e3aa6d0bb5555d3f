"""The bench's multi-rank path on CPU: two gloo ranks (independent replicas) reduce to the slowest
rank's times and the tokens of both; the reference arm runs on rank 0 only."""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
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
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank 1 is slower and has more tokens
        got = bench.reduce_over_ranks(dist, torch.device("cpu"), 1.0 + rank, 2.0 + 3 * rank, 9000 + 500 * rank)
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_two_ranks_reduce_to_slowest_time_and_all_tokens():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    for r in range(world):
        step_ms, e2e_ms, tokens = out[r]
        assert step_ms == 2.0 and e2e_ms == 5.0 and tokens == 9000 + 9500


def test_single_process_passes_through():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(None, None, 1.5, 2.5, 7) == (1.5, 2.5, 7)


def test_reference_arm_under_torchrun_prints_on_rank_0_only():
    env = dict(os.environ, PYTHONPATH=ROOT)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--ref-fraction", "0.0005"]
    res = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1 and '"impl": "reference"' in lines[0]
