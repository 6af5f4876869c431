"""The multi-rank host path of bench.py on CPU: two gloo ranks share the
barrier and take the slowest rank's seconds, and the whole-job value is the
replicas' units over that time (weak scaling, no collective in the data
path).  The reference arm prints from rank 0 only."""
from __future__ import annotations

import importlib.util
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import torch.distributed as dist
    b = _bench()
    barrier, reduce_max = b.collectives(world, "gloo")
    barrier()
    secs = reduce_max(1.0 + 0.5 * rank)  # rank 1 is the slowest
    value = b.weak_scaling_value(8192, 10, world, secs)
    barrier()
    out.put((rank, secs, value))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, secs, value in res:
        assert secs == 1.5
        assert value == pytest.approx(8192 * 2 * 10 / 1.5)


def test_single_rank_collectives_are_no_ops():
    b = _bench()
    barrier, reduce_max = b.collectives(1)
    barrier()
    assert reduce_max(3.25) == 3.25
    assert b.weak_scaling_value(100, 4, 1, 2.0) == 200.0


def test_reference_arm_prints_on_rank_zero_only():
    """Rank 1 of a two-rank reference run exits 0 without output or work."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "1"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
