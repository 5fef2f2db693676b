"""Row entropy and the logprob backward on the GPU, against the oracle.

Entropy (the actor entropy tracked beside the KL, vLLM blog "Finish RL training faster",
section 3.2 results): within the logprob tolerance of the fp64 oracle, logp and logZ
bit-equal to the plain path, and the same invariance (row alone or in a batch, decode
versus prefill, emulated TP split), since it is formed by the same tile tree.

Backward (the pages differentiate a training graph beside the inference forward; it must
be correct, not deterministic; same page, section 3.1): dl = g (onehot - p) is rounded to
bf16 (relative error <= 2^-9) before two fp32-accumulating GEMMs, so every element of dX
and dW must lie within 2^-8 sum |dl| |operand| of the fp64 gradient (twice the rounding
bound; the fp32 error of z and p is below 1e-5 relative), plus 1e-6 of the largest value.
"""
import numpy as np
import pytest
import torch

import oracle
from bit_consistent_logprob_gb300 import (LP_PHASE_DECODE, LP_PHASE_PREFILL, Engine, inputs,
                                          logprobs_with_grad)

from gpu_util import LOGP_TOL, assert_bit_equal, require_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_cuda()


@pytest.mark.parametrize("T,H,V,N", [(300, 256, 4096, 4), (257, 1024, 32001, 8)])
def test_entropy_matches_oracle_and_keeps_logp_bits(dev, T, H, V, N):
    X = inputs.hidden_states(T, H, seed=T, device=dev)
    W = inputs.lm_head(V, H, seed=T, device=dev, std=0.05)
    ids = inputs.uniform_ids(T, V, seed=T, device=dev)
    with Engine(W, n_leaves=N, max_tokens=T) as eng:
        lp, lz, ent = eng.logprobs_entropy(X, ids)
        lp0, lz0 = eng.logprobs(X, ids, return_logZ=True)
        eng.check()
    assert_bit_equal(lp, lp0, "logp with entropy")
    assert_bit_equal(lz, lz0, "logZ with entropy")
    rows = np.unique(np.r_[0, T - 1, np.random.default_rng(T).choice(T, 40)])
    want = oracle.entropy(X.cpu(), W.cpu(), rows=rows)
    got = ent.cpu().double().numpy()[rows]
    err = np.abs(got - want).max()
    assert err <= LOGP_TOL, err
    assert np.all(got >= 0) and np.all(got <= np.log(V) + 1e-4)


def test_entropy_invariance(dev):
    T, H, V, N = 1500, 1024, 32001, 8
    X = inputs.hidden_states(T, H, seed=9, device=dev)
    W = inputs.lm_head(V, H, seed=9, device=dev)
    ids = inputs.uniform_ids(T, V, seed=9, device=dev)
    with Engine(W, n_leaves=N, max_tokens=T) as eng:
        _, _, ent = eng.logprobs_entropy(X, ids)
        for r in (0, 700, T - 1):
            _, _, one = eng.logprobs_entropy(X[r:r + 1], ids[r:r + 1])
            assert_bit_equal(one, ent[r:r + 1], f"row {r} alone")
        for B in (1, 7, 128, 256):
            _, _, dec = eng.logprobs_entropy(X[300:300 + B], ids[300:300 + B], phase=LP_PHASE_DECODE)
            assert_bit_equal(dec, ent[300:300 + B], f"decode B={B}")
        _, _, pre = eng.logprobs_entropy(X[5:1205], ids[5:1205], phase=LP_PHASE_PREFILL)
        assert_bit_equal(pre, ent[5:1205], "shifted batch")
        eng.check()
    for s in (2, 4, 8):
        with Engine(W, n_leaves=N, tp_slices=s, max_tokens=T) as e2:
            _, _, tp = e2.logprobs_entropy(X, ids)
            e2.check()
        assert_bit_equal(tp, ent, f"tp_slices={s}")


def _grad_bounds(dl, W, X):
    bx = (2.0 ** -8) * (np.abs(dl) @ np.abs(W))
    bw = (2.0 ** -8) * (np.abs(dl).T @ np.abs(X))
    return bx, bw


def _bf16_f64(t):
    return t.float().cpu().double().numpy()


@pytest.mark.parametrize("T,H,V,N,chunk", [
    (300, 256, 4001, 4, 300),     # 3 row tiles, ragged vocabulary, one chunk
    (300, 256, 4001, 4, 128),     # three backward chunks accumulate into dW
    (300, 256, 4001, 4, 200),     # a two-row-tile chunk (a CTA pair), then a ragged one
    (97, 512, 32001, 8, 97),      # one partial row tile, leaves of 64
    (130, 384, 1000, 2, 130),     # H not a multiple of the 256-column GEMM tile
])
def test_backward_matches_oracle(dev, T, H, V, N, chunk):
    X = inputs.hidden_states(T, H, seed=T + V, device=dev)
    W = inputs.lm_head(V, H, seed=T + V, device=dev, std=0.05)
    ids = inputs.uniform_ids(T, V, seed=T + V, device=dev)
    g = torch.randn(T, generator=torch.Generator().manual_seed(T), dtype=torch.float32).to(dev)
    with Engine(W, n_leaves=N, max_tokens=T) as eng:
        _, lz = eng.logprobs(X, ids, return_logZ=True)
        eng.backward_reserve(chunk)
        dX, dW = eng.logprobs_backward(X, ids, lz, g)
        eng.check()
    want_dX, want_dW, dl = oracle.logprob_grad(X.cpu(), W.cpu(), ids.cpu().numpy(),
                                               g.cpu().double().numpy())
    bx, bw = _grad_bounds(dl, _bf16_f64(W), _bf16_f64(X))
    ex = np.abs(dX.cpu().double().numpy() - want_dX)
    ew = np.abs(dW.cpu().double().numpy() - want_dW)
    assert np.all(ex <= bx + 1e-6 * np.abs(want_dX).max()), ex.max()
    assert np.all(ew <= bw + 1e-6 * np.abs(want_dW).max()), ew.max()


def test_backward_accumulates_and_skips_outputs(dev):
    T, H, V, N = 200, 256, 4096, 4
    X = inputs.hidden_states(T, H, seed=3, device=dev)
    W = inputs.lm_head(V, H, seed=3, device=dev)
    ids = inputs.uniform_ids(T, V, seed=3, device=dev)
    g = torch.ones(T, device=dev)
    with Engine(W, n_leaves=N, max_tokens=T) as eng:
        _, lz = eng.logprobs(X, ids, return_logZ=True)
        eng.backward_reserve(T)
        dX, dW = eng.logprobs_backward(X, ids, lz, g)
        dX2, none = eng.logprobs_backward(X, ids, lz, g, need_dW=False)
        none2, dW2 = eng.logprobs_backward(X, ids, lz, g, need_dX=False, dW=dW.clone(),
                                           accumulate=True)
        eng.check()
    assert none is None and none2 is None
    assert torch.equal(dX2, dX)
    torch.testing.assert_close(dW2, 2 * dW, rtol=1e-6, atol=1e-7)


def test_autograd_function(dev):
    T, H, V, N = 256, 256, 4096, 4
    X = inputs.hidden_states(T, H, seed=4, device=dev).requires_grad_(True)
    W = inputs.lm_head(V, H, seed=4, device=dev)
    ids = inputs.uniform_ids(T, V, seed=4, device=dev)
    g = torch.linspace(-1, 1, T, device=dev)
    with Engine(W, n_leaves=N, max_tokens=T) as eng:
        Wp = W.requires_grad_(True)
        logp = logprobs_with_grad(eng, X, Wp, ids)
        assert_bit_equal(logp.detach(), eng.logprobs(X.detach(), ids), "autograd forward")
        (logp * g).sum().backward()
        _, lz = eng.logprobs(X.detach(), ids, return_logZ=True)
        dX, dW = eng.logprobs_backward(X.detach(), ids, lz, g.contiguous())
        eng.check()
    assert X.grad.dtype == torch.bfloat16 and Wp.grad.dtype == torch.bfloat16
    torch.testing.assert_close(X.grad, dX.to(torch.bfloat16), rtol=0, atol=0)
    torch.testing.assert_close(Wp.grad, dW.to(torch.bfloat16), rtol=0, atol=0)


def test_backward_qwen_shape_rows(dev):
    # Qwen-shape lm_head (H = 2048, V = 151936): dX of sampled rows against the oracle
    T, H, V, N = 600, 2048, 151936, 8
    X = inputs.hidden_states(T, H, seed=1001, device=dev)
    W = inputs.lm_head(V, H, seed=1001, device=dev)
    ids = inputs.uniform_ids(T, V, seed=1001, device=dev)
    g = torch.randn(T, generator=torch.Generator().manual_seed(5), dtype=torch.float32).to(dev)
    with Engine(W, n_leaves=N, max_tokens=T) as eng:
        _, lz = eng.logprobs(X, ids, return_logZ=True)
        eng.backward_reserve(256)
        dX, _ = eng.logprobs_backward(X, ids, lz, g, need_dW=False)
        eng.check()
    rows = np.array([0, 255, 256, 599])
    Xs = X[rows].cpu()
    want_dX, _, dl = oracle.logprob_grad(Xs, W.cpu(), ids.cpu().numpy()[rows],
                                         g.cpu().double().numpy()[rows])
    bx = (2.0 ** -8) * (np.abs(dl) @ np.abs(_bf16_f64(W)))
    ex = np.abs(dX.cpu().double().numpy()[rows] - want_dX)
    assert np.all(ex <= bx + 1e-6 * np.abs(want_dX).max()), ex.max()


def test_entropy_qwen_shape_rows(dev):
    # Qwen-shape lm_head: entropy of sampled rows of a 2-row-tile batch against the oracle, and
    # the entropy path's logp bits equal to the plain path's at full vocabulary width
    T, H, V, N = 300, 2048, 151936, 8
    X = inputs.hidden_states(T, H, seed=1003, device=dev)
    W = inputs.lm_head(V, H, seed=1003, device=dev)
    ids = inputs.uniform_ids(T, V, seed=1003, device=dev)
    with Engine(W, n_leaves=N, max_tokens=T) as eng:
        lp, lz, ent = eng.logprobs_entropy(X, ids)
        assert_bit_equal(lp, eng.logprobs(X, ids), "logp with entropy at the Qwen shape")
        eng.check()
    rows = np.array([0, 127, 128, 299])
    want = oracle.entropy(X.cpu(), W.cpu(), rows=rows)
    err = np.abs(ent.cpu().double().numpy()[rows] - want).max()
    assert err <= 1e-4, err


def test_backward_qwen_shape_dw_rows(dev):
    # Qwen-shape lm_head (H = 2048, V = 151936), 600 rows in chunks of 256: selected rows of dW
    # (tile edges, the last vocabulary row, and rows that are sampled ids) against an fp64
    # reference dW[v] = sum_t dl[t, v] X[t], with dl[t, v] = g_t (1[v = y_t] - e^(z - logZ_t))
    # from the exact logits and the forward's logZ; the bound allows the bf16 rounding of dl.
    T, H, V, N = 600, 2048, 151936, 8
    X = inputs.hidden_states(T, H, seed=1002, device=dev)
    W = inputs.lm_head(V, H, seed=1002, device=dev)
    ids = inputs.uniform_ids(T, V, seed=1002, device=dev)
    g = torch.randn(T, generator=torch.Generator().manual_seed(6), dtype=torch.float32).to(dev)
    with Engine(W, n_leaves=N, max_tokens=T) as eng:
        _, lz = eng.logprobs(X, ids, return_logZ=True)
        eng.backward_reserve(256)
        _, dW = eng.logprobs_backward(X, ids, lz, g, need_dX=False)
        eng.check()
    ids_h = ids.cpu().numpy()
    vs = np.array(sorted({0, 1, 127, 128, 255, 256, 75000, V - 1, *ids_h[[0, 299, 599]].tolist()}))
    Xd = _bf16_f64(X)                               # [T, H]
    Wd = _bf16_f64(W[torch.as_tensor(vs, device=dev)])  # [S, H]
    z = Xd @ Wd.T                                   # exact-ish fp64 logits [T, S]
    onehot = (ids_h[:, None] == vs[None, :]).astype(np.float64)
    dl = g.cpu().double().numpy()[:, None] * (onehot - np.exp(z - lz.cpu().double().numpy()[:, None]))
    want = dl.T @ Xd                                # [S, H]
    got = dW[torch.as_tensor(vs, device=dev)].cpu().double().numpy()
    bound = (2.0 ** -8) * (np.abs(dl).T @ np.abs(Xd)) + 1e-6 * np.abs(want).max()
    err = np.abs(got - want)
    assert np.all(err <= bound), (err / np.maximum(bound, 1e-30)).max()
