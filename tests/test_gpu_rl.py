"""Acceptance statistics and the REINFORCE Zero loss on the GPU, against the oracle.

Acceptance statistics (vLLM blog "Finish RL training faster", sections 2 and 3.2):
* max |d| is exact: the kernel's max over fp32 |d| must be the fp32 rounding of the
  oracle's exact max (rounding is monotone);
* mean and std of |d| within the fp32 rounding of each d (|d32 - d| <= 2^-24 |d|, and std
  moves by at most max |d32 - d|), plus fp64 summation error;
* k3 within the relative error of the fp32 per-token term; and bit-equal to the D3 of
  lp_importance_weights, which sums the same per-token terms over the same block tree.

REINFORCE Zero (REINFORCE Zero summary, section 4; vLLM blog, section 1):
* advantages are bit-exact (same fp64 operations in the same order);
* gate decisions are exact: the token gate is decided on the fp32 d on both sides, and the
  test data keep every response's log-ratio sum more than 1e-9 from the sequence bounds;
* w_hat and the gradient within 1e-6 relative (fp32 e^d against fp64);
* the loss within 1e-6 of (1/B) sum_i |A_i| max_t w_hat (the fp32 weights' relative error
  bounds each response's term).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from bit_consistent_logprob_gb300 import Engine, LpError, inputs
from bit_consistent_logprob_gb300._native import LP_STAT_COUNT

from gpu_util import assert_bit_equal, require_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return require_cuda()


@pytest.fixture(scope="module")
def eng(dev):
    W = inputs.lm_head(512, 256, seed=3, device=dev)
    e = Engine(W, n_leaves=4, max_tokens=256)
    yield e
    e.close()


def _stats(eng, a, b, mask=None):
    out = eng.acceptance_stats(a, b, mask)
    eng.check()
    v = out.cpu().numpy()
    return dict(max=v[0], mean=v[1], std=v[2], k3=v[3], n_valid=int(v[4]))


def _check_stats(got, want):
    assert got["n_valid"] == want["n_valid"]
    if want["n_valid"] == 0:
        assert got == dict(max=0.0, mean=0.0, std=0.0, k3=0.0, n_valid=0)
        return
    assert got["max"] == float(np.float32(want["max"]))
    eps = 2.0 ** -23
    assert abs(got["mean"] - want["mean"]) <= eps * want["mean"] + 1e-15
    assert abs(got["std"] - want["std"]) <= eps * want["max"] + 1e-12
    assert abs(got["k3"] - want["k3"]) <= 1e-5 * want["k3"] + 1e-15


@pytest.mark.parametrize("T", [0, 1, 1023, 1024, 1025, 300_001, 3_000_000])
def test_acceptance_stats_match_oracle(eng, dev, T):
    lp, lm, mask = inputs.synthetic_is_inputs(T, seed=T + 5, device=dev)
    got = _stats(eng, lp, lm, mask)
    want = oracle.acceptance_stats(lp.cpu().numpy(), lm.cpu().numpy(), mask.cpu().numpy())
    _check_stats(got, want)
    got = _stats(eng, lp, lm)  # no mask: every token valid
    want = oracle.acceptance_stats(lp.cpu().numpy(), lm.cpu().numpy())
    _check_stats(got, want)


def test_k3_is_bit_equal_to_d3(eng, dev):
    lp, lm, mask = inputs.synthetic_is_inputs(2_500_001, seed=11, device=dev)
    stats = eng.acceptance_stats(lp, lm, mask)
    _, d3, nv = eng.importance_weights(lp, lm, mask)
    eng.check()
    assert stats[3].item() == d3.item() and int(stats[4].item()) == nv.item()


def test_acceptance_stats_identical_inputs_are_exactly_zero(eng, dev):
    lp, _, mask = inputs.synthetic_is_inputs(1_000_003, seed=12, device=dev)
    got = _stats(eng, lp, lp.clone(), mask)
    assert (got["max"], got["mean"], got["std"], got["k3"]) == (0.0, 0.0, 0.0, 0.0)
    assert got["n_valid"] == int(mask.sum().item())


def test_acceptance_stats_nan_handling(eng, dev):
    a = torch.tensor([0.0, -1.0, float("nan"), -2.0] * 300, device=dev)
    b = torch.tensor([0.0, -1.5, -3.0, -2.0] * 300, device=dev)
    m = torch.tensor([1, 1, 0, 1] * 300, dtype=torch.uint8, device=dev)
    got = _stats(eng, a, b, m)  # the NaN tokens are masked out
    assert got["max"] == 0.5 and got["n_valid"] == 900
    got = _stats(eng, a, b)
    assert all(math.isnan(got[k]) for k in ("max", "mean", "std", "k3"))


# ---------------------------------------------------------------- REINFORCE Zero
def _rz_inputs(n_groups, G, lo, hi, seed, dev, lag=0.05):
    offs, rewards = inputs.response_batch(n_groups, G, lo, hi, seed)
    T = int(offs[-1])
    lp, lm, mask = inputs.synthetic_is_inputs(T, seed=seed, lag_std=lag, device=dev)
    return lp, lm, mask, offs.to(dev), rewards.to(dev)


MODES = {
    "plain": dict(),
    "tis": dict(tis_cap=1.02),
    "token_gate": dict(token_gate=(-0.02, 0.03)),
    "seq_gate": dict(seq_gate=(-0.4, 0.4)),
    "all": dict(tis_cap=1.05, token_gate=(-0.1, 0.08), seq_gate=(-1.0, 1.0)),
}


def _oracle_kwargs(opts):
    kw, flags = {}, 0
    if "tis_cap" in opts:
        flags |= oracle.TIS
        kw["tis_cap"] = float(np.float32(opts["tis_cap"]))
    if "token_gate" in opts:
        flags |= oracle.TOKEN_GATE
        kw["token_log_lo"], kw["token_log_hi"] = opts["token_gate"]
    if "seq_gate" in opts:
        flags |= oracle.SEQ_GATE
        kw["seq_log_lo"], kw["seq_log_hi"] = opts["seq_gate"]
    kw["flags"] = flags
    return kw


def _check_rz(eng, lp, lm, mask, offs, rewards, G, opts):
    loss, w_hat, grad, adv, n_kept = eng.reinforce_zero(lp, lm, offs, rewards, G, mask=mask,
                                                        **opts)
    eng.check()
    want = oracle.reinforce_zero(lp.cpu().numpy(), lm.cpu().numpy(), offs.cpu().numpy(),
                                 rewards.cpu().numpy(), G, mask=mask.cpu().numpy(),
                                 **_oracle_kwargs(opts))
    if "seq_gate" in opts:
        lo, hi = opts["seq_gate"]
        margin = np.minimum(np.abs(want["seq_logratio"] - lo), np.abs(want["seq_logratio"] - hi))
        assert margin.min() > 1e-9, "test data too close to a sequence-gate bound"
    assert np.array_equal(adv.cpu().numpy(), want["adv"])
    assert n_kept.item() == int(want["kept"].sum())
    w = w_hat.cpu().double().numpy()
    g = grad.cpu().double().numpy()
    assert np.array_equal(w == 0, want["w_hat"] == 0), "a different set of tokens was zeroed"
    assert np.allclose(w, want["w_hat"], rtol=1e-6, atol=0)
    assert np.allclose(g, want["grad"], rtol=1e-6, atol=1e-30)
    B = rewards.shape[0]
    bound = 1e-6 * np.abs(want["adv"]).sum() / B * max(want["w_hat"].max(), 1.0) + 1e-12
    assert abs(loss.item() - want["loss"]) <= bound, (loss.item(), want["loss"])
    return loss, w_hat, grad


@pytest.mark.parametrize("mode", list(MODES))
def test_reinforce_zero_matches_oracle(eng, dev, mode):
    lp, lm, mask, offs, rewards = _rz_inputs(8, 8, 1, 3000, seed=21, dev=dev)
    _check_rz(eng, lp, lm, mask, offs, rewards, 8, MODES[mode])


def test_reinforce_zero_at_importance_weight_workload_scale(eng, dev):
    # 512 responses (64 groups of 8) of U[128, 8192] tokens, the importance-weight workload
    lp, lm, mask, offs, rewards = _rz_inputs(64, 8, 128, 8192, seed=1005, dev=dev)
    assert int(offs[-1]) > 1_500_000
    _check_rz(eng, lp, lm, mask, offs, rewards, 8, {})
    _check_rz(eng, lp, lm, mask, offs, rewards, 8, MODES["all"])


@pytest.mark.parametrize("n_groups", [512, 513, 1025])
def test_reinforce_zero_over_several_chunks_of_responses(eng, dev, n_groups):
    # 2048, 2052 and 4100 short responses: the last block's tree over the response terms
    # takes one full chunk of 2048, a second chunk of four, and three chunks
    lp, lm, mask, offs, rewards = _rz_inputs(n_groups, 4, 1, 40, seed=31 + n_groups, dev=dev)
    assert rewards.shape[0] == 4 * n_groups
    _check_rz(eng, lp, lm, mask, offs, rewards, 4, {})
    _check_rz(eng, lp, lm, mask, offs, rewards, 4, MODES["seq_gate"])


def test_reinforce_zero_degenerate_cases(eng, dev):
    # equal policies: w = 1 and group-centred advantages cancel
    lp, _, mask, offs, rewards = _rz_inputs(4, 4, 1, 50, seed=22, dev=dev)
    mask[offs[:-1]] = 1
    loss, w_hat, _, _, _ = eng.reinforce_zero(lp, lp.clone(), offs, rewards, 4, mask=mask)
    eng.check()
    assert abs(loss.item()) < 1e-15
    assert torch.all(w_hat[mask.bool()] == 1.0)
    # empty responses, an empty batch
    lpe = torch.zeros(0, device=dev)
    loss, _, _, _, kept = eng.reinforce_zero(
        lpe, lpe, torch.zeros(3, dtype=torch.int64, device=dev),
        torch.tensor([1.0, 0.0], device=dev), 2)
    loss0, _, _, _, _ = eng.reinforce_zero(lpe, lpe, torch.zeros(1, dtype=torch.int64, device=dev),
                                           torch.zeros(0, device=dev), 1)
    eng.check()
    assert loss.item() == 0.0 and kept.item() == 2 and loss0.item() == 0.0


def test_reinforce_zero_per_token_outputs_ignore_other_groups(eng, dev):
    lp, lm, mask, offs, rewards = _rz_inputs(6, 4, 1, 400, seed=23, dev=dev)
    opts = MODES["all"]
    loss, w_hat, grad = (t.clone() for t in eng.reinforce_zero(lp, lm, offs, rewards, 4,
                                                               mask=mask, **opts)[:3])
    # move the groups around (same B): every token's w_hat and gradient keep their bits
    order = [3, 0, 5, 1, 4, 2]
    o = offs.cpu()
    seqs = [(int(o[4 * g]), int(o[4 * g + 4])) for g in order]
    idx = torch.cat([torch.arange(a, b) for a, b in seqs]).to(dev)
    lens = torch.tensor([int(o[i + 1] - o[i]) for g in order for i in range(4 * g, 4 * g + 4)])
    offs2 = torch.zeros(25, dtype=torch.int64)
    offs2[1:] = torch.cumsum(lens, 0)
    rw2 = torch.cat([rewards[4 * g:4 * g + 4] for g in order])
    _, w2, g2, _, _ = eng.reinforce_zero(lp[idx], lm[idx], offs2.to(dev), rw2, 4, mask=mask[idx],
                                         **opts)
    eng.check()
    assert_bit_equal(w2, w_hat[idx], "w_hat after moving groups")
    assert_bit_equal(g2, grad[idx], "gradient after moving groups")
    for _ in range(2):  # run to run
        again = eng.reinforce_zero(lp, lm, offs, rewards, 4, mask=mask, **opts)[0]
        assert again.item() == loss.item()


def test_reinforce_zero_rejects_bad_arguments(eng, dev):
    lp, lm, mask, offs, rewards = _rz_inputs(2, 4, 1, 30, seed=24, dev=dev)
    with pytest.raises(LpError):
        eng.reinforce_zero(lp, lm, offs, rewards, 3, mask=mask)  # 3 does not divide 8
    with pytest.raises(LpError):
        eng.reinforce_zero(lp, lm, offs, rewards, 4, mask=mask, tis_cap=0.0)
    with pytest.raises(LpError):
        eng.reinforce_zero(lp, lm, offs, rewards, 4, mask=mask, seq_gate=(1.0, -1.0))
    # a response range past T is reported through the sticky status and read as empty
    bad = offs.clone()
    bad[-1] = int(offs[-1]) + 5
    eng.reinforce_zero(lp, lm, bad, rewards, 4, mask=mask)
    with pytest.raises(LpError, match="token range"):
        eng.check()
    eng.clear_status()
    eng.check()
