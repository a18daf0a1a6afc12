"""The multi-GPU path is replicas only: each rank runs the whole step on its
own GPU and the job's time is the slowest rank's.  These CPU tests run the
host-side logic of that path with two gloo ranks (no GPU)."""

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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # Rank r saw (10 + r) ms for the device-timed steps and (5 (2 - r)) s end to end.
    t = bench.max_over_ranks([10.0 + rank, 5.0 * (2 - rank)], dist)
    v = bench.replica_rate(world, 100, 4, t[0] * 1e-3)
    q.put((rank, t, v))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, t, v in results:
        assert t == [11.0, 10.0]                      # max over ranks, element-wise
        assert v == pytest.approx(2 * 100 * 4 / 11e-3 / 1e9)


def test_single_process_keeps_its_own_times():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.5]) == [3.0, 4.5]
    assert bench.replica_rate(1, 1e9, 2, 1.0) == pytest.approx(2.0)


def test_reference_arm_other_ranks_exit_quietly():
    # Under torchrun only rank 0 runs the reference arm; the others exit 0
    # without work or output.
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
