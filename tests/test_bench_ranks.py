"""Host-side logic of bench.py's multi-process run, on CPU with the gloo backend.

The path is replicas only (no collective on it): N ranks each run the step on
their own GPU, the timed region is reduced with a max over ranks, and the
whole-job value counts every rank's bytes.  These tests run that reduction in
two real processes, and check that the reference arm does no work on ranks
other than 0.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, values, out_q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        got = bench.max_over_ranks(values[rank], dist, torch.device("cpu"))
        out_q.put((rank, got))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_processes():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    values = [3.25, 7.5]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, values, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert res == {0: 7.5, 1: 7.5}


def test_whole_job_value_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.whole_job_value(1e9, 1.0, 1)
    assert one == pytest.approx(1000.0)
    assert bench.whole_job_value(1e9, 1.0, 4) == pytest.approx(4 * one)   # weak scaling: N replicas
    assert bench.whole_job_value(1e9, 2.0, 4) == pytest.approx(2 * one)   # at the slowest rank's time


def test_reference_arm_idle_on_other_ranks():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
