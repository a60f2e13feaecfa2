"""Host logic of the multi-rank benchmark on CPU: two gloo ranks exchange their
timings and byte counts through the same helpers bench.py uses under torchrun
(rank seeds, max and sum over ranks).  No GPU, no data-path collective."""
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
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, _ = bench.dist_env()
        t_ms = 10.0 * (r + 1)                 # rank-specific timing
        nbytes = 1000 * (r + 1)
        mx = bench.max_over_ranks(t_ms, w)
        sm = bench.sum_over_ranks(nbytes, w)
        bench.barrier(w)
        q.put((r, w, mx, sm, bench.rank_seed(7, r)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_timings():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for r, w, mx, sm, seed in got:
        assert w == 2
        assert mx == 20.0                     # the slowest rank's time
        assert sm == 3000.0                   # bytes of both ranks
        assert seed == 7 + 1000 * r           # rank 0 runs the workload's own seed
    assert got[0][4] != got[1][4]


def test_single_rank_helpers_are_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.sum_over_ranks(4.0, 1) == 4.0
    assert bench.rank_seed(3, 0) == 3
