"""The multi-process path of bench.py on the CPU (gloo, world size 2): the
ranks are independent replicas that only meet at the barriers around the
timed region and in the max over ranks of the measured times; the reference
arm runs on rank 0 alone. No GPU is touched."""
import multiprocessing as mp
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


def _rank_main(rank, world, port, times, out):
    os.environ.update(WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.Dist("gloo")
    d.barrier()
    got = d.max(times[rank])
    d.barrier()
    d.close()
    out.put((rank, got))


def test_max_over_ranks_with_gloo():
    world, port = 2, _free_port()
    times = [0.031, 0.045]  # the slower replica decides the job's step time
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 0.045, 1: 0.045}


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    env = dict(os.environ)
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        os.environ.pop(k, None)
    try:
        d = bench.Dist("gloo")
        assert d.dist is None and d.max(1.25) == 1.25
        d.barrier()
        d.close()
    finally:
        os.environ.clear()
        os.environ.update(env)


def test_reference_arm_runs_on_rank_zero_only():
    # a non-zero rank of a torchrun launch exits 0 at once, printing nothing
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
