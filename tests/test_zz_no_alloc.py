"""lp_logprobs_noalloc, called through the C ABI.

This entry point serves callers that cannot call cudaMalloc (code running during CUDA
graph capture, runtimes that plan device memory with their own allocator, hosts that
forbid allocation after start-up): it takes no handle and keeps its scratch in a fixed
file-scope device array.  Two calls in a row must give the same bits as the handle-based
lp_logprobs on the same inputs, and oversized calls must be refused before any work.

This file is collected last so that a run stopping at the first failure has already
run every other test; it also passes when run alone in a fresh process.
"""
import ctypes

import pytest
import torch

from bit_consistent_logprob_gb300 import Engine, _native, inputs
from bit_consistent_logprob_gb300._native import LP_ERR_INVALID_ARG, LP_OK

from gpu_util import assert_bit_equal, require_cuda

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def noalloc(lib, W, X, ids, n_leaves, out, out_logZ):
    T, H = X.shape
    V = W.shape[0]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.lp_logprobs_noalloc(_p(W), H, V, n_leaves, _p(X), X.stride(0), _p(ids), T,
                                   _p(out), _p(out_logZ), stream)


@pytest.mark.parametrize("T,H,V,N", [
    (96, 256, 4096, 4),       # one 96-row tile (96-row X boxes)
    (300, 1024, 32001, 8),    # 3 row tiles, ragged vocabulary tail
    (1, 512, 1000, 2),        # one-token decode row
])
def test_noalloc_matches_handle_path_on_two_calls(T, H, V, N):
    dev = require_cuda()
    lib = _native.load()
    W = inputs.lm_head(V, H, seed=V, device=dev)
    batches = []
    for k in range(2):
        X = inputs.hidden_states(T, H, seed=100 * k + T, device=dev)
        ids = inputs.uniform_ids(T, V, seed=100 * k + T, device=dev)
        batches.append((X, ids))
    with Engine(W, n_leaves=N, max_tokens=T) as eng:
        refs = [eng.logprobs(X, ids, return_logZ=True) for X, ids in batches]
        eng.check()
    outs = []
    for X, ids in batches:  # two calls in a row share the static scratch
        lp = torch.full((T,), float("nan"), device=dev)
        lz = torch.full((T,), float("nan"), device=dev)
        rc = noalloc(lib, W, X, ids, N, lp, lz)
        assert rc == LP_OK, lib.lp_noalloc_last_error()
        outs.append((lp, lz))
    torch.cuda.synchronize()
    for (lp, lz), (ref_lp, ref_lz) in zip(outs, refs):
        assert_bit_equal(lp, ref_lp, "no-alloc logp vs lp_logprobs")
        assert_bit_equal(lz, ref_lz, "no-alloc logZ vs lp_logprobs")


def test_noalloc_refuses_calls_beyond_its_scratch():
    dev = require_cuda()
    lib = _native.load()
    H, V = 256, 151936                      # 2374 log-sum-exp tiles of 64 columns
    W = inputs.lm_head(V, H, seed=1, device=dev)
    T = 442                                 # 442 * 2374 > 2^20 row-tiles
    X = inputs.hidden_states(T, H, seed=1, device=dev)
    ids = inputs.uniform_ids(T, V, seed=1, device=dev)
    out = torch.empty(T, device=dev)
    assert noalloc(lib, W, X, ids, 4, out, None) == LP_ERR_INVALID_ARG
    assert b"static scratch" in lib.lp_noalloc_last_error()
    # the largest call that fits still works and matches the handle path
    rc = noalloc(lib, W, X[:441], ids[:441], 4, out[:441], None)
    assert rc == LP_OK, lib.lp_noalloc_last_error()
    with Engine(W, n_leaves=4, max_tokens=441) as eng:
        ref = eng.logprobs(X[:441], ids[:441])
        eng.check()
    torch.cuda.synchronize()
    assert_bit_equal(out[:441], ref, "largest no-alloc call")
