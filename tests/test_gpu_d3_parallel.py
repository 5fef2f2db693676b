"""D3 and the acceptance statistics of a token stream split across data-parallel ranks,
through the C ABI on one GPU.

D3 is a per-update mean over all valid tokens (REINFORCE Zero summary, section 3), so ranks
that each hold part of the stream must combine their tokens.  The exchange only moves the
fp64 partials of fixed 1024-token blocks (IsoExec summary: collectives transport partials),
then the same fixed tree runs over them.  The ranks are emulated by slices of one stream
(their kernels never wait on one another); the NCCL path runs with a one-rank group.
"""
import os
import socket

import pytest
import torch

from bit_consistent_logprob_gb300 import (Engine, acceptance_stats_data_parallel,
                                          importance_weights_data_parallel, inputs)

from gpu_util import assert_bit_equal, require_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def eng():
    dev = require_cuda()
    W = inputs.lm_head(4096, 256, seed=3, device=dev)
    e = Engine(W, n_leaves=4, max_tokens=64)
    yield e
    e.close()


@pytest.mark.parametrize("bounds,masked", [
    ([0, 1024, 5000], True),
    ([0, 4096, 2_000_896, 3_000_000], True),      # 3 M tokens, a ragged last rank
    ([0, 2048, 2048], False),                      # an empty last rank, no mask
    ([0, 7168], True),                             # one rank
])
def test_split_stream_gives_the_single_call_bits(eng, bounds, masked):
    dev = require_cuda()
    T = bounds[-1]
    lp, lm, mask = inputs.synthetic_is_inputs(T, seed=T, device=dev)
    if not masked:
        mask = None
    w, d3, nv = eng.importance_weights(lp, lm, mask)
    ws, sums, cnts = [], [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        w_r, s_r, c_r = eng.importance_weights_partials(lp[a:b], lm[a:b],
                                                        None if mask is None else mask[a:b])
        assert s_r.shape[0] == (b - a + 1023) // 1024
        ws.append(w_r)
        sums.append(s_r)
        cnts.append(c_r)
    d3_p, nv_p = eng.d3_from_partials(torch.cat(sums), torch.cat(cnts))
    torch.cuda.synchronize()
    eng.check()
    assert_bit_equal(torch.cat(ws), w, "per-token w")
    assert_bit_equal(d3_p, d3, "D3 from gathered block partials")
    assert nv_p.item() == nv.item()


@pytest.mark.parametrize("bounds,nan_at", [
    ([0, 1024, 5000], None),
    ([0, 4096, 2_000_896, 3_000_000], None),
    ([0, 2048, 9000], 7000),                       # a NaN difference on a later rank
])
def test_split_stream_acceptance_statistics(eng, bounds, nan_at):
    dev = require_cuda()
    T = bounds[-1]
    lp, lm, mask = inputs.synthetic_is_inputs(T, seed=T + 1, device=dev)
    if nan_at is not None:
        lp[nan_at] = float("nan")
        mask[nan_at] = 1
    want = eng.acceptance_stats(lp, lm, mask)
    parts = [eng.acceptance_stats_partials(lp[a:b], lm[a:b], mask[a:b])
             for a, b in zip(bounds[:-1], bounds[1:])]
    got = eng.acceptance_stats_from_partials(torch.cat([p[0] for p in parts], dim=1).contiguous(),
                                             torch.cat([p[1] for p in parts]),
                                             torch.cat([p[2] for p in parts]))
    torch.cuda.synchronize()
    eng.check()
    assert_bit_equal(got, want, "statistics from gathered block partials")
    if nan_at is not None:
        assert torch.isnan(got[0]).item()


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def test_data_parallel_helper_with_nccl(eng):
    import torch.distributed as dist

    dev = require_cuda()
    lp, lm, mask = inputs.synthetic_is_inputs(50_000, seed=5, device=dev)
    w, d3, nv = eng.importance_weights(lp, lm, mask)
    st = eng.acceptance_stats(lp, lm, mask)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(_free_port())
    dist.init_process_group("nccl", rank=0, world_size=1)
    try:
        w_p, d3_p, nv_p = importance_weights_data_parallel(eng, lp, lm, mask)
        st_p = acceptance_stats_data_parallel(eng, lp, lm, mask)
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    eng.check()
    assert_bit_equal(w_p, w, "w")
    assert_bit_equal(d3_p, d3, "D3")
    assert nv_p.item() == nv.item()
    assert_bit_equal(st_p, st, "acceptance statistics")
