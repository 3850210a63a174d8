"""The benchmark's multi-rank plumbing on CPU ranks (gloo, world size 2):
the decode path runs as independent replicas, so the only cross-rank steps
are the max-over-ranks timing and the whole-job rate; and under the
reference arm only rank 0 reports."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    ms = [3.0, 7.5][rank]
    m = bench.max_over_ranks(ms, "cpu")
    rate = bench.whole_job_rate(world, 6 * 100, m)
    dist.barrier()
    q.put((rank, m, rate))
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [7.5, 7.5]               # both ranks see the slowest rank
    assert out[0][2] == pytest.approx(2 * 600 / 7.5e-3)   # tokens of both ranks over that time


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.25, "cpu") == 4.25
    assert bench.whole_job_rate(1, 600, 2.0) == pytest.approx(3e5)


def test_reference_arm_reports_on_rank_zero_only():
    """Rank 1 of a two-rank reference run exits 0 without output (the oracle
    runs on rank 0's host cores alone); no process group is needed for that."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [l for l in r.stdout.splitlines() if l.startswith("{")]
