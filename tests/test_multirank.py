"""Rank logic of the benchmark's data-parallel (weak-scaling) path, run as
two gloo ranks on CPU: each rank serves its own sequences, the job's time is
the slowest rank's, throughput counts every rank's tokens, and only rank 0
runs the host-core reference arm."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        local = [3.0, 7.5][rank]
        mx = bench.max_over_ranks(local, "cpu")
        ids = torch.tensor([bench.context_seq_id(b, rank) for b in range(64)], dtype=torch.int64)
        gathered = [torch.empty_like(ids) for _ in range(world)]
        dist.all_gather(gathered, ids)
        distinct = len(set(torch.cat(gathered).tolist())) == 64 * world

        class A:
            steps, warmup = 1, 0
        ref = bench.run_reference(A, rank, world) if rank != 0 else "skipped"
        dist.barrier()
        q.put((rank, mx, distinct, ref))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_and_sharding():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, distinct, ref in res:
        assert mx == 7.5            # max over ranks, seen by every rank
        assert distinct             # no sequence served by two ranks
    assert res[1][3] is None        # rank 1 does no reference work and prints nothing


def test_job_throughput_counts_all_ranks():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.job_tokens_per_s(64, 1, 10, 5.0)
    assert one == pytest.approx(64 * 10 / 5e-3)
    assert bench.job_tokens_per_s(64, 4, 10, 5.0) == pytest.approx(4 * one)
    assert bench.max_over_ranks(1.25, "cpu") == 1.25   # no process group: the local value
