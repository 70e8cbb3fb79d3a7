"""The multi-rank logic of bench.py on CPU: two gloo ranks (no GPU).

bench.py runs one independent replica of the workload per GPU (weak scaling, no collective on
the data path); the only cross-rank steps are the barriers around the timed region, the max of
the per-rank times, and the aggregation of units over ranks.  These run here as two processes
on the gloo backend."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench._dist() == (world, rank, rank)
        bench._barrier(world)
        # per-rank "seconds": the slowest rank decides
        secs = [0.25, 0.75][rank]
        mx = bench.dist_max(secs, world)
        value = bench.aggregate(1000.0, world, mx)
        results[rank] = (mx, value)
        bench._barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time_and_aggregate_units():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
        codes = [p.exitcode for p in procs]
        for p in procs:
            if p.is_alive():
                p.kill()
        assert codes == [0, 0], codes
        got = dict(results)
    # both ranks see the slowest rank's time, and value = units of all ranks / that time
    assert got[0] == got[1] == (0.75, 2000.0 / 0.75)


def test_single_rank_helpers_are_identities():
    import bench

    assert bench.dist_max(1.5, 1) == 1.5
    assert bench.aggregate(300.0, 1, 2.0) == 150.0
    bench._barrier(1)  # no process group needed


def test_reference_arm_runs_on_rank_zero_only():
    import argparse

    import bench

    args = argparse.Namespace(cpu_tokens=8, steps=1, warmup=0)
    assert bench.run_reference(args, world=2, rank=1) is None
