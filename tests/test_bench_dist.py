"""The benchmark's multi-rank path on CPU: two gloo ranks on 127.0.0.1.

Every rank processes its own batch of the same shape (weak scaling, no data
exchange in the pass); the ranks meet only to combine their timings (the
slowest rank's time) and their output voxels (the sum).
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench
    from sparse_voxel_grid_leaf_gb300 import synth
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ijk, off = bench.rank_batch(synth, "pr1_b2_res32", rank)
        ms = 10.0 + 5.0 * rank          # rank 1 is the slowest
        voxels = 1000 * (rank + 1)      # stand-in output sizes
        t, v = bench.job_totals(dist, ms, voxels, "cpu")
        # shape of this rank's batch and a digest of its voxels
        digest = int(np.bitwise_xor.reduce(ijk.astype(np.int64).ravel() * 2654435761 % (1 << 31)))
        out.put((rank, t, v, len(off) - 1, int(len(ijk)), digest))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_combine_time_and_work():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
    for p in procs:
        if p.is_alive():
            p.kill()
            p.join()
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(world))
    for rank, t, v, B, n, _ in res:
        assert t == pytest.approx(15.0)          # max over ranks
        assert v == pytest.approx(3000.0)        # sum over ranks
        assert B == 2                            # same workload shape on every rank
        assert n > 0
    # independent batches: the ranks' voxels differ
    assert res[0][5] != res[1][5] or res[0][4] != res[1][4]


def test_single_process_totals():
    import bench
    assert bench.job_totals(None, 12.5, 7, "cpu") == (12.5, 7.0)
