"""The bench's multi-rank path on the host, with world_size-2 gloo process
groups on the CPU: the cross-rank maximum that sets a job's time, the
whole-job throughput, and the reference arm's rank rule (rank 0 alone
prints its line, the other ranks exit 0 without work)."""

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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r reports times 10 + r and 5 - r: the job takes the slowest
        got = bench.max_over_ranks([10.0 + rank, 5.0 - rank], "cpu")
        dist.barrier()
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert out[0] == out[1] == [11.0, 5.0]


def test_max_over_ranks_without_a_group_is_the_identity():
    assert not dist.is_initialized()
    assert bench.max_over_ranks([1.5, 2.0], "cpu") == [1.5, 2.0]


def test_job_throughput_counts_every_rank():
    # two ranks of 16384 tokens each, the slowest taking 0.5 ms
    assert bench.job_tokens_per_s(16384, 2, 0.5) == pytest.approx(65536000.0)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
