"""bench.py under a multi-process launch, on CPU: the GPU arm refuses to run on more than one
GPU before touching CUDA, and the reference arm (the CPU oracle) runs on rank 0 alone while
the other ranks exit without work."""
import argparse
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from conftest import ROOT


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
        args = argparse.Namespace(config=1, steps=1, warmup=3, ref_budget=0.0, temperature=0.0,
                                  seed=1)
        ref = bench.run_reference(args, rank, world)
        dist.barrier()
        out.put((rank, None if ref is None else ref["impl"]))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_reference_arm_runs_on_rank0_only():
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
    assert res == [(0, "reference"), (1, None)]


@pytest.mark.timeout(120)
@pytest.mark.parametrize("env,argv", [({"WORLD_SIZE": "2", "RANK": "0"}, []),
                                      ({"WORLD_SIZE": "2", "RANK": "1"}, []),
                                      ({}, ["--gpus", "2"])])
def test_gpu_arm_refuses_more_than_one_gpu(env, argv):
    """Exit status 2 and a message, before any CUDA call: a poisoned CUDA_VISIBLE_DEVICES
    and a missing library would make any later step fail differently."""
    full = dict(os.environ, **env, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "1", *argv],
                       capture_output=True, text=True, env=full, timeout=100)
    assert r.returncode == 2, (r.returncode, r.stderr[-2000:])
    assert "exactly one GPU" in r.stderr
    assert r.stdout.strip() == ""
