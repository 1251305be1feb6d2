"""Multi-process host logic of the benchmark, on CPU with the gloo backend
(world size 2). The forward has no exchange step: ranks run independent
batches (weak scaling) and only the timing is reduced, max over ranks.
"""
from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        # Each rank timed its own steps; the job's time is the slowest rank's.
        t = bench.max_over_ranks(0.5 + rank)
        bench.barrier()
        gbs = bench.whole_job_gbs(1000, 10, world, t)
        # The reference arm prints from rank 0 only; other ranks exit without work.
        rc = bench.main(["--impl", "reference", "--steps", "1", "--warmup", "1"]) if rank else 0
        out.put((rank, t, gbs, rc))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, t, gbs, rc in got:
        assert t == pytest.approx(1.5)
        assert gbs == pytest.approx(1000 * 10 * 2 / 1.5 / 1e9)
        assert rc == 0


def test_single_process_helpers_are_identity():
    import bench
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.whole_job_gbs(2_000_000_000, 3, 1, 2.0) == pytest.approx(3.0)
