"""bench.py's multi-GPU path, run on the CPU as two gloo ranks.

The step does not shard: with N GPUs every rank runs its own replica of the whole step and no
collective enters the timed work.  What the ranks share is the bookkeeping around it: the
rank/world read from the launcher's environment, the barrier around the timed region, the
maximum over ranks of each timing (the slowest replica sets the step time) and the value, which
counts the units of every rank.  The reference arm runs on rank 0 only.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, queue):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    r, w, local = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    try:
        # per-rank step and decode times: rank 1 has the slower step, rank 0 the slower decode
        mine = [1e-3 * (1 + rank), 4e-4 * (2 - rank)]
        dist.barrier()
        step, dec = bench.max_over_ranks(dist, mine)
        value = bench.replica_throughput(w, 64, step)
        dist.barrier()
        queue.put((rank, (r, w, local), step, dec, value))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_replica_and_count_all_units():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        results = sorted(queue.get(timeout=180) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0, 0]
    for rank, env, step, dec, value in results:
        assert env == (rank, 2, rank)
        assert step == 2e-3
        assert dec == 8e-4
        assert value == 2 * 64 / 2e-3


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(None, [3.0, 1.5]) == [3.0, 1.5]
    assert bench.replica_throughput(1, 64, 0.5) == 128.0


def test_reference_arm_runs_on_rank_zero_only(capsys):
    class Args:
        workload = bench.DEFAULT_WORKLOAD
        steps = 1
        warmup = 0
    assert bench.run_reference(Args(), rank=1, world=2) is None
    assert capsys.readouterr().out == ""
