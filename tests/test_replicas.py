"""The N>1 bench path is N independent replicas: the only cross-rank traffic is
the barrier and the max-over-ranks of the elapsed time, and rank 0 alone
reports.  Checked with two gloo ranks on the CPU (no GPU)."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        t = bench.max_over_ranks(10.0 + 5.0 * rank, world)
        class A:  # the reference arm's arguments
            steps, warmup = 1, 0
        ref = bench.run_reference(A, world, rank) if rank != 0 else "skipped"
        out.put((rank, t, ref))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_and_only_rank0_reports():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [15.0, 15.0]      # both ranks see the max
    assert res[1][2] is None                        # non-zero ranks print nothing
