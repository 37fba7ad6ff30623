"""bench.py's multi-rank host logic on CPU with two gloo ranks: the timing reduction is
the max over ranks, and the reference arm runs on rank 0 only."""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.rank_env() == (world, rank, rank)
        vals = bench.max_over_ranks([1.0 + rank, 10.0 - rank, 0.5 * rank], "cpu")
        class Args:
            steps, warmup = 1, 3
        ref = bench.reference_arm(Args(), rank, world) if rank != 0 else "rank0-skipped"
        out.put((rank, vals, ref))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_reference_rank_gate():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    results = dict()
    for _ in range(world):
        rank, vals, ref = out.get(timeout=120)
        results[rank] = (vals, ref)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in range(world):
        assert results[rank][0] == [2.0, 10.0, 0.5]
    assert results[1][1] is None          # non-zero ranks do no reference work


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.5], "cpu") == [3.0, 4.5]
