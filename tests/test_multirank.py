"""The multi-rank path of bench.py on CPU (gloo, world size 2).

Ranks are replicas: the whole-job time is the slowest rank's (max over ranks)
and the value counts every rank's bytes; the reference arm runs on rank 0
only and the other ranks exit without work.
"""

import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        secs = 2.0 if rank == 1 else 1.0          # rank 1 is the slow one
        slowest = bench.max_over_ranks(secs, world, "cpu")
        q.put((rank, slowest, bench.whole_job_gbs(10**9, 5, world, slowest)))
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank_and_all_bytes():
    import torch.multiprocessing as mp
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
    for rank, slowest, gbs in out:
        assert slowest == 2.0
        assert gbs == pytest.approx(10**9 * 5 * 2 / 2.0 / 1e9)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.whole_job_gbs(473497600, 10, 1, 1.0) == pytest.approx(4.734976)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
