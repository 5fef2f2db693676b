"""Vocabulary-parallel lm_head, through the C ABI on one GPU.

Ranks that each hold a slice of the lm_head's rows compute the (max, sum-exp) partials of
their vocabulary tiles and the sampled logit of the rows whose token they own; the partials
are moved (never combined by the transport) and the fixed tile tree finishes them (IsoExec
summary, "Parallelism-invariant kernels": collectives only transport partials).  Ranks are
emulated by handles over slices of one W; the NCCL helper runs with a one-rank group.
"""
import os
import socket

import pytest
import torch

from bit_consistent_logprob_gb300 import Engine, inputs, logprobs_vocab_parallel

from gpu_util import assert_bit_equal, require_cuda

pytestmark = pytest.mark.gpu

H, N = 1024, 8


@pytest.mark.parametrize("cuts,V,T", [
    ([0, 12800, 25600], 32001, 300),     # three slices, the last one ragged
    ([0, 16384], 32001, 256),            # two slices; 256 rows: two row tiles
    ([0, 128, 4096], 8000, 7),           # a one-tile slice; a decode batch
])
def test_vocab_split_gives_the_full_lm_head_bits(cuts, V, T):
    dev = require_cuda()
    W = inputs.lm_head(V, H, seed=V, device=dev)
    X = inputs.hidden_states(T, H, seed=T, device=dev)
    ids = inputs.uniform_ids(T, V, seed=T + V, device=dev)
    with Engine(W, n_leaves=N, max_tokens=T) as full:
        want, wantZ = full.logprobs(X, ids, return_logZ=True)
        full.check()
    bounds = cuts + [V]
    ms_parts, zy_parts = [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        with Engine(W[a:b], n_leaves=N, max_tokens=T) as part:
            ms, zy = part.vocab_partials(X, ids - a)
            # the sampled logit of a row this slice owns; NaN for rows owned elsewhere
            inside = (ids >= a) & (ids < b)
            assert torch.isfinite(zy[inside]).all() and torch.isnan(zy[~inside]).all()
            ms_parts.append(ms.clone())
            zy_parts.append(zy.clone())
            part.check()
    ms_all = torch.cat(ms_parts, dim=0).contiguous()
    starts = torch.tensor(cuts, dtype=torch.int64, device=dev)
    owner = torch.searchsorted(starts, ids.to(torch.int64), right=True) - 1
    zy_all = torch.stack(zy_parts)[owner, torch.arange(T, device=dev)].contiguous()
    with Engine(W[:128], n_leaves=N, max_tokens=T) as fin:   # lends its status word only
        got, gotZ = fin.logprobs_from_vocab_partials(V, ms_all, zy_all, ids, return_logZ=True)
        fin.check()
    assert_bit_equal(got, want, "logp from vocabulary partials")
    assert_bit_equal(gotZ, wantZ, "logZ from vocabulary partials")


def test_misaligned_slice_is_refused_before_any_collective():
    dev = require_cuda()
    W = inputs.lm_head(4096, H, seed=2, device=dev)
    with Engine(W[64:], n_leaves=N, max_tokens=8) as e:
        X = inputs.hidden_states(8, H, seed=2, device=dev)
        ids = inputs.uniform_ids(8, 4096, seed=2, device=dev)
        with pytest.raises(ValueError):
            logprobs_vocab_parallel(e, X, ids, 64, 4096)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def test_vocab_parallel_helper_with_nccl():
    import torch.distributed as dist

    dev = require_cuda()
    V, T = 32001, 200
    W = inputs.lm_head(V, H, seed=9, device=dev)
    X = inputs.hidden_states(T, H, seed=9, device=dev)
    ids = inputs.uniform_ids(T, V, seed=9, device=dev)
    with Engine(W, n_leaves=N, max_tokens=T) as eng:
        want, wantZ = eng.logprobs(X, ids, return_logZ=True)
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(_free_port())
        dist.init_process_group("nccl", rank=0, world_size=1)
        try:
            got, gotZ = logprobs_vocab_parallel(eng, X, ids, 0, V, return_logZ=True)
            torch.cuda.synchronize()
        finally:
            dist.destroy_process_group()
        eng.check()
    assert_bit_equal(got, want, "logp")
    assert_bit_equal(gotZ, wantZ, "logZ")
