"""The bench's multi-rank host logic on CPU ranks (gloo, world size 2): the
timed work of each replica is aggregated as the slowest rank's time, the
job's throughput counts every rank's tokens, and under torchrun the
reference arm prints one line from rank 0 while the other ranks exit 0."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as tmp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    ms = [12.5, 30.0][rank]
    slowest = bench.max_over_ranks(ms, world, "cpu")
    q.put((rank, slowest, bench.job_throughput(world, 64, 10, slowest)))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_throughput_gloo():
    world = 2
    port = _free_port()
    q = tmp.get_context("spawn").SimpleQueue()
    tmp.start_processes(_worker, args=(world, port, q), nprocs=world, start_method="spawn")
    got = sorted(q.get() for _ in range(world))
    for rank, slowest, tput in got:
        assert slowest == 30.0
        assert tput == pytest.approx(2 * 64 * 10 / 0.030)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(7.0, 1, "cpu") == 7.0
    assert bench.job_throughput(1, 1, 100, 10.0) == pytest.approx(10000.0)


@pytest.mark.slow
def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    env = dict(os.environ, OMP_NUM_THREADS="1")
    out = subprocess.run(
        [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
         "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
         "--impl", "reference", "--config", "tiny", "--gpus", "2", "--steps", "2", "--warmup", "1"],
        capture_output=True, text=True, timeout=600, env=env, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
