"""Multi-process checks on the CPU (gloo, world size 2 and 4).

* bench.py's N > 1 path runs one replica per rank: the ranks meet only at the timing
  barriers and reduce the step time with a max; rank 0 reports the aggregate.
* The tensor-parallel split of K: rank r owns the contiguous leaves [r*N/s, (r+1)*N/s),
  reduces them to its node of the fixed leaf tree, and the nodes are only moved (an
  all-gather, no reducing collective) before the upper levels of the same tree are applied
  (IsoExec blog summary, "Parallelism-invariant kernels").  The result must equal the
  single-process tree bit for bit, which is what the GPU's emulated split relies on.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _init(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)


def _bench_worker(rank, world, port, out):
    import sys

    sys.path.insert(0, ROOT)
    import bench

    _init(rank, world, port)
    bench.barrier(dist)
    ms = bench.max_over_ranks(dist, 10.0 + rank, torch.device("cpu"))
    bench.barrier(dist)
    out[rank] = ms
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_bench_replicas_take_the_slowest_rank(world):
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_bench_worker, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn")
    assert [out[r] for r in range(world)] == [10.0 + world - 1] * world


def _tp_worker(rank, world, port, n_leaves, seed, out):
    import sys

    sys.path.insert(0, ROOT)
    import oracle as orc

    _init(rank, world, port)
    rng = np.random.default_rng(seed)
    # fp32 leaf partials for 64 logits; every rank sees the same data and owns a slice
    P = (rng.standard_normal((64, n_leaves)) * np.exp2(rng.integers(-20, 20, (64, n_leaves))))
    P = P.astype(np.float32)
    per = n_leaves // world
    mine = orc.tree_fp32(P[:, rank * per:(rank + 1) * per])          # this rank's tree node
    gathered = [torch.empty(64, dtype=torch.float32) for _ in range(world)]
    dist.all_gather(gathered, torch.from_numpy(mine.copy()))          # data movement only
    nodes = torch.stack(gathered, dim=1).numpy()
    top = orc.tree_fp32(nodes)                                        # upper levels
    if rank == 0:
        out["split"] = top.view(np.int32).tolist()
        out["whole"] = orc.tree_fp32(P).view(np.int32).tolist()
    dist.destroy_process_group()


@pytest.mark.parametrize("world,n_leaves", [(2, 8), (4, 8), (2, 4), (4, 4)])
def test_tp_leaf_split_over_ranks_is_bit_exact(world, n_leaves):
    oracle.build()
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_tp_worker, args=(world, _free_port(), n_leaves, 7 + world, out),
                       nprocs=world, start_method="spawn")
    assert out["split"] == out["whole"]
