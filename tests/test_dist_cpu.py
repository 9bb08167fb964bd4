"""The benchmark's multi-rank path on CPU: two gloo ranks (one process each),
the rendezvous through the environment variables torchrun sets, the
slowest-rank timing reduction and the reference arm's rank-0-only rule."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    ws, r, local = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=ws)
    try:
        slowest = bench.max_over_ranks(10.0 * (rank + 1), "cpu")
        # the reference arm: every rank but 0 returns before any work
        import types
        args = types.SimpleNamespace(gpus=world, steps=1, warmup=0)
        ran = None
        if rank != 0:
            ran = bench.run_reference(args)
        out[rank] = (ws, r, local, slowest, ran)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert sorted(res) == [0, 1]
    for rank, (ws, r, local, slowest, ran) in res.items():
        assert (ws, r, local) == (world, rank, rank)
        assert slowest == 20.0
        assert ran is None


def test_single_process_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
