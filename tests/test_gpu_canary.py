"""Canary-padded outputs: no call writes outside the buffers it is given.

Every device output is the middle of a larger buffer whose margins hold a canary bit pattern;
after the call (and a check of the sticky status) the margins must be bit-for-bit unchanged.
Shapes are ragged (partial row tiles, a vocabulary that is not a multiple of 64 or 128) so
that every tail path of every kernel runs.
"""
import pytest
import torch

from bit_consistent_logprob_gb300 import Engine, inputs

from gpu_util import require_cuda

pytestmark = pytest.mark.gpu

PAD = 1024
CANARY = 0x7FC0DEAD


def padded(n, dtype, dev):
    """(full buffer, middle view of n elements) with the margins set to the canary."""
    elem = torch.tensor([], dtype=dtype).element_size()
    words = (n * elem + 3) // 4 + 2 * PAD
    raw = torch.full((words,), CANARY, dtype=torch.int32, device=dev)
    start = PAD * 4 // elem
    return raw, raw.view(dtype)[start:start + n]


def check_margins(raw, n, dtype, what):
    elem = torch.tensor([], dtype=dtype).element_size()
    end_word = PAD + (n * elem + 3) // 4
    head = raw[:PAD].cpu()
    tail = raw[end_word:].cpu()
    assert torch.all(head == CANARY), f"{what}: write before the buffer"
    assert torch.all(tail == CANARY), f"{what}: write after the buffer"


@pytest.mark.parametrize("T,H,V,N,fp8", [(333, 256, 4001, 4, False), (1, 512, 1000, 2, False),
                                         (333, 512, 4001, 4, True)])
def test_logprob_outputs_stay_in_bounds(T, H, V, N, fp8):
    dev = require_cuda()
    X = inputs.hidden_states(T, H, seed=T, device=dev)
    W = inputs.lm_head(V, H, seed=T, device=dev)
    ids = inputs.uniform_ids(T, V, seed=T, device=dev)
    with Engine(W, n_leaves=N, max_tokens=128, fp8=fp8) as eng:  # several row chunks
        raw_lp, lp = padded(T, torch.float32, dev)
        raw_lz, lz = padded(T, torch.float32, dev)
        eng.logprobs(X, ids, out=lp, out_logZ=lz)
        if not fp8:
            raw_e, ent = padded(T, torch.float32, dev)
            eng.logprobs_entropy(X, ids, out=lp, out_logZ=lz, out_entropy=ent)
        eng.check()
        torch.cuda.synchronize()
    check_margins(raw_lp, T, torch.float32, "logp")
    check_margins(raw_lz, T, torch.float32, "logZ")
    if not fp8:
        check_margins(raw_e, T, torch.float32, "entropy")
    assert torch.isfinite(lp).all()


def test_rl_outputs_stay_in_bounds():
    dev = require_cuda()
    W = inputs.lm_head(512, 256, seed=1, device=dev)
    offs, rewards = inputs.response_batch(3, 4, 1, 900, seed=2)
    T, B = int(offs[-1]), rewards.numel()
    lp, lm, mask = inputs.synthetic_is_inputs(T, seed=3, device=dev)
    with Engine(W, n_leaves=4, max_tokens=64) as eng:
        raw_w, w = padded(T, torch.float32, dev)
        raw_d3, d3 = padded(1, torch.float64, dev)
        raw_nv, nv = padded(1, torch.int64, dev)
        eng.importance_weights(lp, lm, mask, out_w=w, out_d3=d3, out_nvalid=nv)
        raw_st, st = padded(5, torch.float64, dev)
        eng.acceptance_stats(lp, lm, mask, out=st)
        raw_wh, wh = padded(T, torch.float32, dev)
        raw_g, g = padded(T, torch.float32, dev)
        raw_a, adv = padded(B, torch.float64, dev)
        eng.reinforce_zero(lp, lm, offs.to(dev), rewards.to(dev), 4, mask=mask, tis_cap=1.05,
                           seq_gate=(-2.0, 2.0), out_w_hat=wh, out_grad=g, out_adv=adv)
        eng.check()
        torch.cuda.synchronize()
    for raw, n, dt, what in ((raw_w, T, torch.float32, "w"), (raw_d3, 1, torch.float64, "D3"),
                             (raw_nv, 1, torch.int64, "n_valid"), (raw_st, 5, torch.float64, "stats"),
                             (raw_wh, T, torch.float32, "w_hat"), (raw_g, T, torch.float32, "grad"),
                             (raw_a, B, torch.float64, "advantages")):
        check_margins(raw, n, dt, what)


def test_backward_outputs_stay_in_bounds():
    dev = require_cuda()
    T, H, V, N = 201, 256, 4001, 4
    X = inputs.hidden_states(T, H, seed=5, device=dev)
    W = inputs.lm_head(V, H, seed=5, device=dev)
    ids = inputs.uniform_ids(T, V, seed=5, device=dev)
    g = torch.ones(T, device=dev)
    with Engine(W, n_leaves=N, max_tokens=T) as eng:
        _, lz = eng.logprobs(X, ids, return_logZ=True)
        eng.backward_reserve(64)  # four chunks, the last one partial
        raw_dx, dX = padded(T * H, torch.float32, dev)
        raw_dw, dW = padded(V * H, torch.float32, dev)
        eng.logprobs_backward(X, ids, lz, g, dX=dX.view(T, H), dW=dW.view(V, H))
        eng.check()
        torch.cuda.synchronize()
    check_margins(raw_dx, T * H, torch.float32, "dX")
    check_margins(raw_dw, V * H, torch.float32, "dW")
    assert torch.isfinite(dX).all() and torch.isfinite(dW).all()
