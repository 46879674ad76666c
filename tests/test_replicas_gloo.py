"""Multi-rank host logic of the benchmark on CPU: two gloo ranks.

The path shards into independent batches (replicas, no exchange), so the
ranks meet only in the benchmark: distinct seeded batches per rank, the
slowest rank's time for the job, the whole-job rate from all ranks' rows, and
an oracle arm that only rank 0 runs.
"""
import os
import socket
import sys
import types

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, queue):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from sparse_paged_decode_gb300 import workloads as W

        cpu = torch.device("cpu")
        # per-rank timings: rank r took (10 + r) ms for the steps, (30 - r) end to end
        times = bench.max_over_ranks([10.0 + rank, 30.0 - rank], world, cpu)
        w = W.config(1, seed=bench.batch_seed(1, rank))
        q_sum = float(w.q.float().sum())
        args = types.SimpleNamespace(config=1, steps=1, warmup=0)
        ref = bench.run_reference(args, rank, world) if rank != 0 else "rank 0 not run here"
        torch.distributed.barrier()
        queue.put((rank, times, q_sum, ref))
    finally:
        torch.distributed.destroy_process_group()


def test_two_replicas_meet_only_in_timing():
    world = 2
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, queue)) for r in range(world)]
    for p in procs:
        p.start()
    results = {}
    try:
        for _ in range(world):
            rank, times, q_sum, ref = queue.get(timeout=120)
            results[rank] = (times, q_sum, ref)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    # the slowest rank sets both times, on every rank
    assert results[0][0] == results[1][0] == [11.0, 30.0]
    # each rank has its own batch
    assert results[0][1] != results[1][1]
    # the oracle arm returns nothing (does no work) off rank 0
    assert results[1][2] is None


def test_job_rate_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench

    # 16 rows per rank, 2 ranks, 3 steps in 6 ms -> 16000 rows/s
    assert bench.job_rate(16, 2, 3, 6.0) == pytest.approx(16 * 2 * 3 / 6e-3)
    assert bench.batch_seed(2, 0) != bench.batch_seed(2, 1)
