"""The benchmark's multi-process host logic on the CPU: N processes are N
independent replicas (each computes the whole workload; no data-path
collective), the reported time is the slowest rank's, and the whole-job value
is N times one replica's work over that time.  Two gloo ranks on 127.0.0.1."""
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


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(times[rank], dist, torch.device("cpu"))
        dist.barrier()
        out.put((rank, got, bench.whole_job_throughput(world, 4.0e12, got)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank():
    world, port = 2, free_port()
    times = [5.5, 6.25]
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(out.get(timeout=10) for _ in range(world))
    assert [r[1] for r in res] == [6.25, 6.25]
    assert all(abs(r[2] - 2 * 4.0e12 / 6.25e-3 / 1e12) < 1e-9 for r in res)


def test_one_process_needs_no_collective():
    assert bench.max_over_ranks(3.0, None, None) == 3.0
    assert bench.whole_job_throughput(1, 4.083e12, 4.83) == pytest.approx(845.3, rel=1e-3)


def test_reference_arm_on_a_nonzero_rank_does_no_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
