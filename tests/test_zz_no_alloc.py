"""lp_logprobs_noalloc, called through the C ABI.

This entry point serves callers that cannot call cudaMalloc (runtimes that plan device
memory with their own allocator, hosts that forbid allocation after start-up): it takes no
handle and keeps its scratch in a fixed file-scope device array.  Two calls in a row must
give the same bits as the handle-based lp_logprobs on the same inputs, oversized calls must
be refused before any work, and errors found on the GPU must show in the outputs (NaN),
since this entry point has no status word a caller can read.

This file is collected last so that a run stopping at the first failure has already
run every other test; it also passes when run alone in a fresh process.
"""
import ctypes
import os
import subprocess
import sys

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


def test_noalloc_reports_a_bad_id_on_its_row_only():
    dev = require_cuda()
    lib = _native.load()
    T, H, V, N = 40, 256, 4096, 4
    W = inputs.lm_head(V, H, seed=5, device=dev)
    X = inputs.hidden_states(T, H, seed=5, device=dev)
    ids = inputs.uniform_ids(T, V, seed=5, device=dev)
    with Engine(W, n_leaves=N, max_tokens=T) as eng:
        ref, refZ = eng.logprobs(X, ids, return_logZ=True)
        eng.check()
    bad = ids.clone()
    bad[7] = V          # outside [0, V)
    bad[31] = -1
    lp = torch.empty(T, device=dev)
    lz = torch.empty(T, device=dev)
    assert noalloc(lib, W, X, bad, N, lp, lz) == LP_OK, lib.lp_noalloc_last_error()
    torch.cuda.synchronize()
    assert torch.isnan(lp[[7, 31]]).all()
    keep = torch.ones(T, dtype=torch.bool, device=dev)
    keep[[7, 31]] = False
    assert_bit_equal(lp[keep], ref[keep], "no-alloc logp of the good rows")
    assert_bit_equal(lz, refZ, "no-alloc logZ (it does not depend on the id)")
    # the next call with good ids is clean again: nothing of the bad call is left over
    assert noalloc(lib, W, X, ids, N, lp, lz) == LP_OK
    torch.cuda.synchronize()
    assert_bit_equal(lp, ref, "no-alloc logp after a bad call")


_TIMEOUT_CHILD = r"""
import ctypes, sys, torch
sys.path.insert(0, sys.argv[1])
from bit_consistent_logprob_gb300 import _native, inputs
lib = _native.load()
dev = torch.device("cuda:0")
T, H, V, N = 33, 256, 4096, 4
W = inputs.lm_head(V, H, seed=3, device=dev)
X = inputs.hidden_states(T, H, seed=3, device=dev)
ids = inputs.uniform_ids(T, V, seed=3, device=dev)
lp = torch.zeros(T, device=dev)
lz = torch.zeros(T, device=dev)
s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
for _ in range(2):
    rc = lib.lp_logprobs_noalloc(ctypes.c_void_p(W.data_ptr()), H, V, N,
                                 ctypes.c_void_p(X.data_ptr()), H, ctypes.c_void_p(ids.data_ptr()),
                                 T, ctypes.c_void_p(lp.data_ptr()), ctypes.c_void_p(lz.data_ptr()), s)
    assert rc == 0, lib.lp_noalloc_last_error()
    torch.cuda.synchronize()
    assert torch.isnan(lp).all() and torch.isnan(lz).all(), (lp, lz)
print("all rows NaN")
"""


def test_noalloc_timeout_turns_every_row_into_nan():
    # The test hook marks every call of this process as if one of its bounded waits had
    # expired (no wait is made to run out on the GPU); the caller must then see NaN in
    # every row of logp and logZ.  The hook is read once per process, so it runs in a child.
    require_cuda()
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, LP_TEST_NOALLOC_MARK_TIMEOUT="1")
    out = subprocess.run([sys.executable, "-c", _TIMEOUT_CHILD, root], env=env,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stdout + out.stderr
    assert "all rows NaN" in out.stdout
