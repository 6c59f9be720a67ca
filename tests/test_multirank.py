"""Two-rank host logic of bench.py on CPU (gloo): every rank runs its own replica, ranks
meet only at barriers and at the max-over-ranks timing, and only rank 0 reports."""
import argparse
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world, timeout=__import__("datetime").timedelta(seconds=60))
    try:
        mine = 1.5 + 2.0 * rank                      # each rank's own time
        slowest = bench.max_over_ranks(mine, dist, "cpu")
        dist.barrier()
        args = argparse.Namespace(config=1, steps=1, warmup=3, ref_budget=0.0)
        ref = bench.run_reference(args, rank, world) if rank != 0 else "rank0-skipped"
        out.put((rank, slowest, ref))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_ranks_take_the_slowest_time_and_only_rank0_reports():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=100) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [3.5, 3.5]        # max over ranks on every rank
    assert res[1][2] is None                        # the reference arm: rank 1 does no work


def test_single_process_helpers():
    import bench
    assert bench.max_over_ranks(2.0, None, "cpu") == 2.0
    assert bench.job_throughput(4, 100, 0.5) == 800.0
