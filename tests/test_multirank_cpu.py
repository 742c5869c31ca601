"""N>1 bench path on CPU: world_size-2 gloo ranks (replicas only).

The path shards with no exchange, so the only cross-rank step in bench.py is
the max-over-ranks timing reduction; the reference arm prints on rank 0 only.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    got = bench.max_over_ranks(1.5 + rank)
    out[rank] = got
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_reference_arm_prints_on_rank0_only():
    import argparse

    import bench
    args = argparse.Namespace(workload="tiny", variant="w4a8", steps=1, warmup=0, m=1, k=512,
                              n=256, cpu_budget=0.5, impl="reference", api="grouped",
                              fused=False, path="auto")
    assert bench.run_reference(args, rank=1, world=2) is None
    res = bench.run_reference(args, rank=0, world=2)
    assert res["impl"] == "reference" and res["value"] > 0
    assert res["e2e"]["h2d_bytes_per_step"] == 0 and res["cpu_baseline"]["kind"] == "oracle"
    assert res["config"] == bench.workload_config(args)
