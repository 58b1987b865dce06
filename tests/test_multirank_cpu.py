"""The multi-rank plumbing of bench.py on CPU: two gloo ranks over 127.0.0.1.  The layer
step shards by request and head with no exchange, so N GPUs run N replicas; what crosses
ranks is only the timing reduction (the job's time is its slowest rank's) and the sum of
the units processed."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, local = bench.dist_env()
    d = bench.dist_init(w, "gloo")
    try:
        ms = [3.0, 5.0][rank]          # per-rank step time
        units = [64 * 69, 64 * 69][rank]
        slowest = bench.max_over_ranks(ms, d)
        total = bench.sum_over_ranks(units, d)
        q.put((rank, r, w, local, slowest, total))
    finally:
        d.barrier()
        d.destroy_process_group()


def test_two_rank_reduction_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, (r, rr, w, local, slowest, total) in enumerate(got):
        assert (r, rr, w, local) == (rank, rank, 2, rank)
        assert slowest == 5.0
        assert total == 2 * 64 * 69


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.dist_init(1, "gloo") is None
    assert bench.max_over_ranks(2.5, None) == 2.5
    assert bench.sum_over_ranks(7, None) == 7.0
