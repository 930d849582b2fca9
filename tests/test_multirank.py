"""Several ranks on the CPU (gloo, world size 2): the host side of
``bench.py --gpus N``.  The path does not shard: every rank runs its own
replica of the workload, the job is timed by its slowest rank, and the
value counts the work of all ranks.  The reference arm runs on rank 0 only."""
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = 100.0 + 25.0 * rank          # rank 1 is the slow one
        slowest = bench.max_over_ranks(elapsed, "cpu")
        value = bench.job_tflops(world, 1e12, 10, slowest)
        dist.barrier()
        out.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_replicas_are_timed_by_the_slowest_rank():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()   # both ranks rendezvous on it
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(out.get(timeout=10) for _ in range(world))
    for rank, slowest, value in res:
        assert slowest == 125.0
        # 2 ranks x 1e12 FLOP x 10 steps in 125 ms
        assert value == pytest.approx(2 * 1e12 * 10 / 0.125 / 1e12)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
    assert bench.job_tflops(1, 2e12, 4, 1000.0) == pytest.approx(8.0)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "3", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
