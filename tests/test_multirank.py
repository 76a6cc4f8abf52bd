"""The bench's multi-rank host logic on CPU (gloo, world size 2): each rank
runs its own batch (replicas), the barrier holds, and the whole-job value is
all ranks' tokens over the slowest rank's time (no GPU)."""
import os
import socket
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        sys.path.insert(0, ROOT)
        import bench
        bench.barrier(ws)
        tokens = [100.0, 50.0][rank]
        ms = [2.0, 3.0][rank]
        out[rank] = bench.aggregate(tokens, ms, ws)
        bench.barrier(ws)
    finally:
        dist.destroy_process_group()


def test_replicas_aggregate_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank, args=(2, _free_port(), out), nprocs=2, start_method="spawn")
        res = dict(out)
    for rank in (0, 1):
        tokens, ms, rate = res[rank]
        assert tokens == 150.0 and ms == 3.0       # sum of tokens, slowest rank's time
        assert abs(rate - 150.0 / 3e-3) < 1e-6


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate(7, 2.0, 1) == (7.0, 2.0, 3500.0)
