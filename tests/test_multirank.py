"""The multi-process (one rank per GPU) path's host logic, on CPU with the
gloo backend and two ranks: the timed region is the slowest rank's, the
reported rate counts every rank's units, and under torchrun the reference
arm runs on rank 0 only (the other ranks exit at once, without work)."""
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


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = 10.0 + 5.0 * rank             # rank 1 is the slower one
    ms = bench.slowest_rank_ms(local_ms, dist)
    dist.barrier()
    q.put((rank, ms, bench.whole_job_rate(world, 1024 * 100, ms)))
    dist.destroy_process_group()


def test_two_ranks_slowest_time_and_whole_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, rate in got:
        assert ms == 15.0                     # both ranks see the slowest rank's time
        assert rate == pytest.approx(2 * 1024 * 100 / 0.015)


def test_single_process_keeps_local_time():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank_ms(12.5, None) == 12.5
    assert bench.whole_job_rate(1, 1000, 10.0) == pytest.approx(1000 / 0.010)


def test_reference_arm_nonzero_rank_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-500:]
    assert r.stdout.strip() == ""
