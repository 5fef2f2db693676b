"""Failure detection without a GPU fault.

Every pipeline wait in the kernels is bounded (a %globaltimer budget).  The self-test kernel
waits on an mbarrier that nothing ever arrives on -- a flag that nothing sets -- with that
same bounded wait; it must give up, raise the sticky timeout status and return.  A test hook
makes the leaf GEMM's own abort path run: its copy producer stops early, and the kernel must
drain and return with a timeout status.  The host
reads the status (LP_ERR_TIMEOUT), clears it, and the context keeps working bit-exactly.
Bad sampled ids are the other device-side failure: NaN for that row and LP_ERR_INVALID_ARG.
"""
import time

import pytest
import torch

from bit_consistent_logprob_gb300 import Engine, LpError, inputs
from bit_consistent_logprob_gb300._native import LP_ERR_INVALID_ARG, LP_ERR_TIMEOUT

from gpu_util import assert_bit_equal, require_cuda

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    dev = require_cuda()
    X = inputs.hidden_states(300, 256, seed=2, device=dev)
    W = inputs.lm_head(4096, 256, seed=2, device=dev)
    ids = inputs.uniform_ids(300, 4096, seed=2, device=dev)
    with Engine(W, n_leaves=4, max_tokens=300) as eng:
        before = eng.logprobs(X, ids).clone()
        eng.check()
        t0 = time.perf_counter()
        eng.selftest_wait_timeout(20_000)  # 20 ms budget
        with pytest.raises(LpError) as err:
            eng.check()
        elapsed = time.perf_counter() - t0
        assert err.value.code == LP_ERR_TIMEOUT
        assert 0.015 < elapsed < 5.0, elapsed
        eng.clear_status()
        eng.check()
        after = eng.logprobs(X, ids)
        eng.check()
    assert_bit_equal(after, before, "after a reported timeout")


@pytest.mark.parametrize("T", [100, 300])   # one CTA per tile; CTA pairs (two row-tile pairs)
def test_leaf_gemm_abort_path_reports_timeout_and_recovers(T, monkeypatch):
    # The test hook stops the leaf GEMM's copy producer after its first pipeline stage, as if
    # its own wait had run out.  That stage's copies land and are consumed; the MMA warp's wait
    # for the next stage then runs out, it raises the abort flag (in a pair, the partner's too)
    # and drains its MMAs; the epilogue warps see the flag and stop; the producer's drain finds
    # its one stage complete; TMEM is freed and the kernel returns with nothing in flight.  The
    # host reads LP_ERR_TIMEOUT, and afterwards the context gives the reference bits.
    dev = require_cuda()
    X = inputs.hidden_states(T, 256, seed=5, device=dev)
    W = inputs.lm_head(4096, 256, seed=5, device=dev)
    ids = inputs.uniform_ids(T, 4096, seed=5, device=dev)
    with Engine(W, n_leaves=4, max_tokens=T) as eng:
        ref = eng.logprobs(X, ids).clone()
        eng.check()
    monkeypatch.setenv("LP_WAIT_TIMEOUT_MS", "50")
    monkeypatch.setenv("LP_TEST_STOP_AFTER_STAGES", "1")
    with Engine(W, n_leaves=4, max_tokens=T) as hooked:
        t0 = time.perf_counter()
        hooked.logprobs(X, ids)
        with pytest.raises(LpError) as err:
            hooked.check()
        elapsed = time.perf_counter() - t0
        assert err.value.code == LP_ERR_TIMEOUT
        assert 0.04 < elapsed < 10.0, elapsed
        hooked.clear_status()
        hooked.check()
    monkeypatch.delenv("LP_TEST_STOP_AFTER_STAGES")
    monkeypatch.delenv("LP_WAIT_TIMEOUT_MS")
    with Engine(W, n_leaves=4, max_tokens=T) as eng:
        again = eng.logprobs(X, ids)
        eng.check()
    assert_bit_equal(again, ref, "after the abort path ran")


def test_fp8_leaf_gemm_abort_path_reports_timeout_and_recovers(monkeypatch):
    # The block-FP8 kernel issues its MMAs from two warps (alternate 128-K blocks, each with its
    # own TMEM buffer), and each drains only the MMAs it issued.  With the copy producer stopped
    # after its first block: that block lands, the first MMA warp issues it and the epilogue
    # reads it; both MMA warps' waits for their next blocks run out, they raise the abort flag
    # and drain; the epilogue stops on the flag; the producer's drain finds its copy complete;
    # TMEM is freed with nothing in flight.  The host reads LP_ERR_TIMEOUT, and afterwards the
    # context gives the reference bits.
    dev = require_cuda()
    T, H, V = 200, 512, 4096
    X = inputs.hidden_states(T, H, seed=6, device=dev)
    W = inputs.lm_head(V, H, seed=6, device=dev)
    ids = inputs.uniform_ids(T, V, seed=6, device=dev)
    with Engine(W, n_leaves=4, max_tokens=T, fp8=True) as eng:
        ref = eng.logprobs(X, ids).clone()
        eng.check()
    monkeypatch.setenv("LP_WAIT_TIMEOUT_MS", "50")
    monkeypatch.setenv("LP_TEST_STOP_AFTER_STAGES", "1")
    with Engine(W, n_leaves=4, max_tokens=T, fp8=True) as hooked:
        t0 = time.perf_counter()
        hooked.logprobs(X, ids)
        with pytest.raises(LpError) as err:
            hooked.check()
        elapsed = time.perf_counter() - t0
        assert err.value.code == LP_ERR_TIMEOUT
        assert 0.04 < elapsed < 10.0, elapsed
        hooked.clear_status()
        hooked.check()
    monkeypatch.delenv("LP_TEST_STOP_AFTER_STAGES")
    monkeypatch.delenv("LP_WAIT_TIMEOUT_MS")
    with Engine(W, n_leaves=4, max_tokens=T, fp8=True) as eng:
        again = eng.logprobs(X, ids)
        eng.check()
    assert_bit_equal(again, ref, "after the FP8 abort path ran")


def test_bad_id_is_reported_and_isolated():
    dev = require_cuda()
    X = inputs.hidden_states(200, 256, seed=3, device=dev)
    W = inputs.lm_head(4096, 256, seed=3, device=dev)
    ids = inputs.uniform_ids(200, 4096, seed=3, device=dev)
    with Engine(W, n_leaves=4, max_tokens=200) as eng:
        good = eng.logprobs(X, ids).clone()
        bad = ids.clone()
        bad[17] = 4096
        bad[150] = -1
        lp = eng.logprobs(X, bad)
        with pytest.raises(LpError) as err:
            eng.check()
        assert err.value.code == LP_ERR_INVALID_ARG
        eng.clear_status()
    assert torch.isnan(lp[17]) and torch.isnan(lp[150])
    keep = torch.ones(200, dtype=torch.bool, device=dev)
    keep[[17, 150]] = False
    assert_bit_equal(lp[keep], good[keep], "rows with valid ids")


@pytest.mark.parametrize("buffer", ["ws_ms", "zy", "stat_max", "is_stage", "host_scalars", "wq"])
def test_allocation_failure_is_reported_and_cleaned_up(buffer, monkeypatch):
    # the test hook fails one named workspace allocation; lp_init must return LP_ERR_OOM,
    # free what it had allocated, and a later init must succeed
    dev = require_cuda()
    from bit_consistent_logprob_gb300._native import LP_ERR_OOM

    W = inputs.lm_head(4096, 256, seed=4, device=dev)
    free0 = torch.cuda.mem_get_info()[0]
    monkeypatch.setenv("LP_TEST_FAIL_ALLOC", buffer)
    for _ in range(3):
        with pytest.raises(LpError) as err:
            Engine(W, n_leaves=2, max_tokens=4096, fp8=True)
        assert err.value.code == LP_ERR_OOM and buffer in str(err.value)
    monkeypatch.delenv("LP_TEST_FAIL_ALLOC")
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] >= free0 - (64 << 20)  # nothing leaked
    X = inputs.hidden_states(64, 256, seed=4, device=dev)
    ids = inputs.uniform_ids(64, 4096, seed=4, device=dev)
    with Engine(W, n_leaves=2, max_tokens=4096, fp8=True) as eng:
        assert torch.isfinite(eng.logprobs(X, ids)).all()
        eng.check()
