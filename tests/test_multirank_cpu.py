"""The multi-rank host logic of bench.py on CPU: two gloo ranks on 127.0.0.1.

The scan shards by independent problems (each rank scans its own batch; no collective on
the data path), so what the ranks share is only the timing: every rank's elapsed time is
reduced to the maximum, and the whole-job throughput counts every rank's elements over that
maximum. The ranks' problems must be independent (different seeds) and rank 0's must be the
workload itself.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench
from selective_state_space_diagonal_b300 import workloads as wl


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_seconds = 1.0 + rank          # rank 1 is the slow one
        slowest = bench.reduce_max(local_seconds)
        bench.barrier()
        value = bench.aggregate_value(1000, steps=10, world=world, max_seconds=slowest)
        w = bench.rank_workload(wl.WORKLOADS["trap_bf16_batch"], rank)
        out.put((rank, bench.rank_info(), slowest, value, w.seed))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_timing_and_get_independent_problems():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    base = wl.WORKLOADS["trap_bf16_batch"]
    for rank, (r, ws, lr), slowest, value, seed in results:
        assert (r, ws, lr) == (rank, world, rank)
        assert slowest == 2.0                                  # max over ranks, seen by every rank
        assert value == pytest.approx(1000 * 10 * 2 / 2.0 / 1e9)  # all ranks' elements / slowest
    seeds = [seed for *_, seed in results]
    assert seeds[0] == base.seed and seeds[1] != base.seed


def test_single_process_is_a_no_op_reduction():
    assert bench.reduce_max(3.5) == 3.5
    assert bench.rank_workload(wl.WORKLOADS["euler_f32_tiny"], 0) is wl.WORKLOADS["euler_f32_tiny"]
