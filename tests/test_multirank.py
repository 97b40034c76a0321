"""The replica (N > 1) host path of bench.py on CPU: two gloo ranks on
127.0.0.1. Each rank runs the whole workload on its own GPU, so the only
exchange is the timing: the job's time is the slowest rank's and its
throughput the units of all ranks over that time."""
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, elapsed, units, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out.put((rank,) + bench.reduce_timing(elapsed[rank], units, world))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("elapsed", [(10.0, 15.0), (7.5, 2.5)])
def test_reduce_timing_two_gloo_ranks(elapsed):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, elapsed, 300, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    slowest = max(elapsed)
    for rank, ms, value in res:
        assert ms == slowest
        assert value == pytest.approx(2 * 300 / (slowest / 1000.0))


def test_reduce_timing_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_timing(4.0, 100, 1) == (4.0, 100 / 0.004)


def test_reference_arm_other_ranks_exit_quietly():
    """Under torchrun only rank 0 times the oracle; rank 1 exits 0 and prints nothing."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "3", "--warmup", "3"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
