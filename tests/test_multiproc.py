"""Multi-process checks on the CPU (gloo, world size 2 and 4).

* bench.py's N > 1 path runs one replica per rank: the ranks meet only at the timing
  barriers and reduce the step time with a max; rank 0 reports the aggregate.
* The tensor-parallel split of K: rank r owns the contiguous leaves [r*N/s, (r+1)*N/s),
  reduces them to its node of the fixed leaf tree, and the nodes are only moved (an
  all-gather, no reducing collective) before the upper levels of the same tree are applied
  (IsoExec blog summary, "Parallelism-invariant kernels").  The result must equal the
  single-process tree bit for bit, which is what the GPU's emulated split relies on.
* D3 over a token stream split across ranks: each rank's fp64 partials over 1024-token
  blocks are all-gathered in rank order (moved, never added), so every rank holds the whole
  stream's blocks and the same fixed tree gives one D3 for any number of ranks (REINFORCE
  Zero summary, section 3: a per-update mean over tokens).
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


def _stream_blocks(T, seed):
    """The D3 terms of one synthetic token stream (oracle) and its fp64 sums and valid counts
    per 1024-token block, by plain numpy."""
    rng = np.random.default_rng(seed)
    lp = np.log(rng.uniform(1e-6, 1.0, T)).astype(np.float32)
    lm = (lp + rng.normal(0.0, 0.05, T)).astype(np.float32)
    mask = (rng.uniform(size=T) < 0.9).astype(np.uint8)
    _, term, _, _ = oracle.importance_weights(lp, lm, mask)
    term = np.where(mask != 0, term, 0.0)
    nb = (T + 1023) // 1024
    sums = np.array([term[b * 1024:(b + 1) * 1024].sum() for b in range(nb)])
    cnts = np.array([int(mask[b * 1024:(b + 1) * 1024].sum()) for b in range(nb)], dtype=np.int64)
    return sums, cnts


def _d3_worker(rank, world, port, bounds, seed, out):
    import sys

    sys.path.insert(0, ROOT)
    from bit_consistent_logprob_gb300 import gather_block_partials

    _init(rank, world, port)
    sums, cnts = _stream_blocks(bounds[-1], seed)
    b0, b1 = bounds[rank] // 1024, (bounds[rank + 1] + 1023) // 1024   # this rank's blocks
    s_all, c_all = gather_block_partials(torch.from_numpy(sums[b0:b1].copy()),
                                         torch.from_numpy(cnts[b0:b1].copy()))
    rows = np.stack([sums, -sums, 2 * sums])                # a [3, nb] array of partials
    (r_all,) = gather_block_partials(torch.from_numpy(rows[:, b0:b1].copy()))
    out[rank] = (s_all.numpy().view(np.int64).tolist(), c_all.numpy().tolist(),
                 r_all.numpy().view(np.int64).tolist())
    dist.destroy_process_group()


@pytest.mark.parametrize("bounds", [[0, 3072, 7000], [0, 1024, 9216, 9300]])
def test_d3_block_partials_gather_in_rank_order(bounds):
    # Ranks hold consecutive token ranges, all but the last a multiple of 1024 tokens, with
    # different block counts; every rank must end with the whole stream's blocks, bit for bit,
    # so the same fixed tree over them gives one D3 for any number of ranks.
    world = len(bounds) - 1
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_d3_worker, args=(world, _free_port(), bounds, 17, out), nprocs=world,
                       start_method="spawn")
    sums, cnts = _stream_blocks(bounds[-1], 17)
    rows = np.stack([sums, -sums, 2 * sums])
    for r in range(world):
        assert out[r][0] == sums.view(np.int64).tolist(), f"rank {r} sums"
        assert out[r][1] == cnts.tolist(), f"rank {r} counts"
        assert out[r][2] == rows.view(np.int64).tolist(), f"rank {r} [3, nb] rows"


def _misaligned_worker(rank, world, port, out):
    import sys

    sys.path.insert(0, ROOT)
    from bit_consistent_logprob_gb300 import importance_weights_data_parallel

    _init(rank, world, port)
    if rank == 0:  # not the last rank, and 1000 tokens is not a multiple of 1024
        x = torch.zeros(1000)
        try:
            importance_weights_data_parallel(None, x, x)   # rejected before any collective
            out[rank] = "accepted"
        except ValueError:
            out[rank] = "rejected"
    dist.destroy_process_group()


def test_d3_data_parallel_rejects_a_misaligned_rank():
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_misaligned_worker, args=(2, _free_port(), out), nprocs=2,
                       start_method="spawn")
    assert out[0] == "rejected"


def _vocab_worker(rank, world, port, starts, V_full, T, out):
    import sys

    sys.path.insert(0, ROOT)
    from bit_consistent_logprob_gb300 import gather_vocab_partials

    _init(rank, world, port)
    v0, v1 = starts[rank], (starts[rank + 1] if rank + 1 < world else V_full)
    t0, t1 = v0 // 64, (v1 + 63) // 64                      # this rank's 64-column tiles
    tiles = torch.arange(t0, t1, dtype=torch.float32)
    ms = torch.stack([tiles[:, None] * 1000 + torch.arange(T, dtype=torch.float32),
                      -tiles[:, None].expand(-1, T)], dim=-1)   # [tiles, T, 2], tile-coded
    zy = torch.full((T,), float(rank)) + torch.arange(T, dtype=torch.float32) / 1000
    ids = (torch.arange(T, dtype=torch.int64) * 7919 % V_full).to(torch.int32)
    ms_all, zy_all = gather_vocab_partials(ms, zy, ids, v0, v1 - v0, V_full)
    out[rank] = (ms_all.numpy().tolist(), zy_all.numpy().tolist())
    dist.destroy_process_group()


def test_vocab_partials_gather_in_vocabulary_order_and_pick_the_owner():
    # Three ranks own vocabulary slices starting at multiples of 128; every rank must get
    # all tiles in vocabulary order and, per row, the sampled logit of the rank owning its id.
    starts, V_full, T = [0, 1280, 2560], 4001, 16
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_vocab_worker, args=(3, _free_port(), starts, V_full, T, out), nprocs=3,
                       start_method="spawn")
    nt = (V_full + 63) // 64
    ids = np.arange(T) * 7919 % V_full
    owner = np.searchsorted(np.array(starts), ids, side="right") - 1
    for r in range(3):
        ms_all = np.array(out[r][0])
        assert ms_all.shape == (nt, T, 2)
        assert np.array_equal(ms_all[:, :, 1], -np.arange(nt)[:, None] * np.ones((1, T)))
        assert np.array_equal(ms_all[:, :, 0], np.arange(nt)[:, None] * 1000 + np.arange(T))
        want_zy = owner.astype(np.float32) + np.arange(T, dtype=np.float32) / 1000
        assert np.array_equal(np.array(out[r][1], dtype=np.float32), want_zy), f"rank {r}"
