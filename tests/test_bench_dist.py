"""The multi-process path of bench.py on the CPU (gloo, world size 2): the
max-over-ranks timing reduction, the whole-job throughput, and the reference
arm on ranks other than 0. bench.py runs one replica per GPU with no
data-path collective; these are the only cross-rank steps it has."""
import json
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


def _worker(rank, world, port, queue):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank, world)  # rank 1 is the slow one
        dist.barrier()
        queue.put((rank, slowest))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert codes == [0, 0], codes
    got = dict(queue.get(timeout=5) for _ in range(2))
    assert got == {0: 15.0, 1: 15.0}


def test_single_rank_reduction_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_job_throughput_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.job_gbs(1, 11_448_320, 1000, 20.0)
    assert one == pytest.approx(11_448_320 * 1000 / 0.020 / 1e9)
    # weak scaling: N ranks each doing the same work in the same (max) time
    assert bench.job_gbs(4, 11_448_320, 1000, 20.0) == pytest.approx(4 * one)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "1"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""  # rank 0 alone prints the line
