"""Two CPU ranks on gloo: the data-parallel split of the path and the bench's
max-over-ranks timing reduction.

Each rank takes a contiguous token shard (whole documents of a packed batch),
computes its RMSNorm weight gradient with the oracle, and the ranks sum them
with one all-reduce: the result equals the oracle's dW over the whole batch
(the only cross-shard quantity of the path).  The bench's ``reduce_max`` and
``barrier`` helpers run across the same two ranks.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    import oracle
    from rmsnorm_fwd_bwd_03_gb300.workload import lognormal_doc_lengths
    try:
        dist.init_process_group("gloo", rank=rank, world_size=world)
        rng = np.random.default_rng(0)
        lengths = lognormal_doc_lengths(3000, seed=3)
        cu = np.concatenate([[0], np.cumsum(lengths)])
        T, H, eps = int(cu[-1]), 24, 1e-5
        h = rng.normal(size=(T, H))
        dy = rng.normal(size=(T, H))
        # split on a document boundary near the middle
        cut = int(cu[np.searchsorted(cu, T // 2)])
        lo, hi = (0, cut) if rank == 0 else (cut, T)
        part = torch.tensor(oracle.rmsnorm_dw(dy[lo:hi], h[lo:hi], eps))
        dist.all_reduce(part, op=dist.ReduceOp.SUM)
        full = oracle.rmsnorm_dw(dy, h, eps)
        ok_dw = bool(np.allclose(part.numpy(), full, rtol=1e-12, atol=1e-12))
        bench.barrier(world)
        mx = bench.reduce_max(float(rank + 1) * 1.5, world)
        q.put((rank, ok_dw, mx))
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


def test_two_rank_dw_allreduce_and_timing_max():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ok_dw, mx in res:
        assert ok_dw, f"rank {rank}: sum of shard dW differs from the full dW"
        assert mx == pytest.approx(3.0)
