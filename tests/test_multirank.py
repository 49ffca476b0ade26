"""The benchmark's multi-rank host logic on CPU (two gloo ranks, no GPU).

bench.py under torchrun runs one independent replica per GPU: no data-path
collective, only a barrier around the timed region and the maximum of the
ranks' times; the whole-job value counts what every rank processed.  The
reference arm runs on rank 0 only.
"""
import importlib.util
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    bench = _bench()
    w, r, local = bench.dist_setup()
    dist.init_process_group("gloo", rank=r, world_size=w)
    try:
        dist.barrier()
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, w, "cpu")  # rank 1 is the slow one
        out[rank] = (w, r, local, ms, bench.job_rate(1000.0, 4, w, ms))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_count_both_ranks_work():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        w, r, local, ms, rate = res[rank]
        assert (w, r, local) == (world, rank, rank)
        assert ms == 15.0                       # every rank reports the slowest rank's time
        assert rate == pytest.approx(1000.0 * 4 * world / 0.015)


def test_single_rank_needs_no_process_group():
    bench = _bench()
    assert bench.max_over_ranks(7.5, 1) == 7.5
    assert bench.job_rate(10.0, 3, 1, 2.0) == pytest.approx(15000.0)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert p.returncode == 0, p.stderr
    assert p.stdout.strip() == ""
