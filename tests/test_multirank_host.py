"""The benchmark's multi-rank bookkeeping on CPU ranks (gloo, world size 2): the timed
region is the slowest rank's, the whole-job rates count every rank's work, and the
reference arm runs on rank 0 alone.  (One GPU per rank runs N independent replicas; the
path has no collective of its own.)"""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    w, r, local = bench.dist_setup(None)
    ms = 10.0 + 5.0 * rank                      # rank 1 is the slower one
    t = bench.max_over_ranks(ms, w, "cpu")
    gbs, rows = bench.whole_job_rates(1e9, 32, 100, w, t)
    q.put((r, w, local, t, gbs, rows))
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_every_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for r, (rank, world, local, t, gbs, rows) in enumerate(got):
        assert (rank, world, local) == (r, 2, r)
        assert t == 15.0                          # the slower rank's 15 ms, on both ranks
        assert abs(gbs - 2 * 1e9 * 100 / 0.015 / 1e9) < 1e-6
        assert abs(rows - 2 * 32 * 100 / 0.015) < 1e-6


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun every rank but 0 exits at once, printing nothing."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--gpus", "2", "--steps", "1", "--warmup", "0"],
                         capture_output=True, text=True, env=env, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]
    assert res.stdout.strip() == ""
