"""bench.py's multi-rank path on CPU: world_size 2 over gloo (127.0.0.1).
The benchmark runs one independent replica per rank; the only cross-rank
steps are the barriers around the timed region and the max over ranks of the
elapsed time, and the reference arm runs on rank 0 alone."""
import os
import sys
import types

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank) and dist.get_backend() == "gloo"
    bench.barrier(w)
    slowest = bench.max_over_ranks(10.0 + rank, w, torch.device("cpu"))
    # the reference arm prints from rank 0 only; other ranks return at once
    other = bench.reference_arm(types.SimpleNamespace(), w, r, local, []) if r != 0 else None
    out[rank] = (slowest, other)
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_rank_barrier_and_max_over_ranks():
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
        assert dict(out) == {0: (11.0, None), 1: (11.0, None)}
