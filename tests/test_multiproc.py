"""The multi-GPU bench path on CPU: two gloo ranks on 127.0.0.1.

With one simulated job per GPU (replicas; the simulated ranks never cross
GPUs), the only cross-process steps are the barrier and the max of the timed
region over ranks.  Here two CPU processes check that every rank receives the
slowest rank's time and that the whole-job value counts both replicas; and
that the reference arm prints only on rank 0."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
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
        ms = 10.0 + 5.0 * rank                      # rank 1 is the slow one
        slow = bench.slowest_rank_ms(ms, dist, "cpu")
        dist.barrier()
        q.put((rank, slow, bench.job_gbs(world, 1 << 30, 100, slow)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[1] for g in got] == [15.0, 15.0]
    want = 2 * (1 << 30) * 100 / 15e-3 / 1e9
    assert all(abs(g[2] - want) < 1e-9 * want for g in got)


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0
    assert p.stdout.strip() == ""
