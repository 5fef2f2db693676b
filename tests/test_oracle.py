"""Pins for the fp64 CPU oracle (runs without a GPU).

Each check ties the oracle to something other than itself: exact rational
arithmetic on bf16 inputs (Fraction), a high-precision log-sum-exp written
independently with ``decimal``, closed forms (two-token vocabulary, uniform
logits, shift invariance, one dominant logit), invariants (probabilities sum to
one, D3 = 0 at w = 1, term >= 0) and hand-derived golden values under
``tests/golden/``.  The mutation tests at the end plant plausible mistakes in a
copy of the oracle source and check that the pins catch them.
"""
import math
import os
import shutil
import subprocess
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import pytest

import oracle

getcontext().prec = 60


# ----------------------------------------------------------------- helpers
def f32_to_bf16_bits(a) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest even) and return the uint16 bit patterns."""
    u = np.ascontiguousarray(np.asarray(a, dtype=np.float32)).view(np.uint32).astype(np.uint64)
    rounding = ((u >> 16) & 1) + 0x7FFF
    return ((u + rounding) >> 16).astype(np.uint16)


def bits_to_fraction(b) -> Fraction:
    f = np.array([int(b) << 16], dtype=np.uint32).view(np.float32)[0]
    return Fraction(float(f))


def rand_bf16(shape, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return f32_to_bf16_bits(rng.standard_normal(shape).astype(np.float32) * scale)


def exact_logits(X, W):
    T, H = X.shape
    V = W.shape[0]
    Xf = [[bits_to_fraction(X[t, k]) for k in range(H)] for t in range(T)]
    Wf = [[bits_to_fraction(W[v, k]) for k in range(H)] for v in range(V)]
    return [[sum(Xf[t][k] * Wf[v][k] for k in range(H)) for v in range(V)] for t in range(T)]


def dec(fr: Fraction) -> Decimal:
    return Decimal(fr.numerator) / Decimal(fr.denominator)


def decimal_logprob(zrow, y):
    """log softmax(z)[y] from exact logits, by the unshifted definition in 60-digit decimal."""
    total = sum((dec(z).exp() for z in zrow), Decimal(0))
    return float(dec(zrow[y]) - total.ln()), float(total.ln())


# ----------------------------------------------------------------- logits
def test_logits_exact_rational():
    X = rand_bf16((3, 16), 1)
    W = rand_bf16((5, 16), 2, 0.3)
    z = oracle.logits(X, W)
    ex = exact_logits(X, W)
    for t in range(3):
        for v in range(5):
            assert z[t, v] == pytest.approx(float(ex[t][v]), rel=1e-15, abs=1e-300)


def test_logits_rows_subset_and_orientation():
    # Non-square shapes catch a transposed operand; the row subset must index X rows.
    X = rand_bf16((6, 12), 3)
    W = rand_bf16((4, 12), 4)
    full = oracle.logits(X, W)
    sub = oracle.logits(X, W, rows=[5, 0, 3])
    assert full.shape == (6, 4)
    np.testing.assert_array_equal(sub, full[[5, 0, 3]])
    ex = exact_logits(X, W)
    assert full[5, 2] == pytest.approx(float(ex[5][2]), rel=1e-15)


# ----------------------------------------------------------------- logprobs
def test_logprobs_brute_force_decimal():
    X = rand_bf16((4, 8), 5)
    W = rand_bf16((7, 8), 6, 0.8)
    ids = np.array([0, 6, 3, 1], dtype=np.int32)
    logp, logZ = oracle.logprobs(X, W, ids)
    ex = exact_logits(X, W)
    for t in range(4):
        lp, lz = decimal_logprob(ex[t], int(ids[t]))
        assert logp[t] == pytest.approx(lp, abs=1e-13)
        assert logZ[t] == pytest.approx(lz, abs=1e-13)


def test_two_token_vocab_closed_form():
    # V = 2: log p_y = -log1p(exp(z_other - z_y)).
    X = rand_bf16((5, 6), 7)
    W = rand_bf16((2, 6), 8, 2.0)
    ex = exact_logits(X, W)
    for y in (0, 1):
        ids = np.full(5, y, dtype=np.int32)
        logp, _ = oracle.logprobs(X, W, ids)
        for t in range(5):
            d = float(ex[t][1 - y] - ex[t][y])
            assert logp[t] == pytest.approx(-math.log1p(math.exp(d)), abs=1e-14)


def test_uniform_logits_give_minus_log_v():
    V, H = 4096, 32
    X = rand_bf16((9, H), 9)
    row = rand_bf16((1, H), 10)
    W = np.repeat(row, V, axis=0)
    ids = np.random.default_rng(11).integers(0, V, 9).astype(np.int32)
    logp, _ = oracle.logprobs(X, W, ids)
    np.testing.assert_allclose(logp, -math.log(V), rtol=0, atol=1e-12)


def test_shift_invariance_through_a_constant_column():
    # Append a hidden column with x = 1 and w = c for every token: every logit moves by c,
    # so logZ moves by c and every logprob is unchanged.
    X = rand_bf16((4, 10), 12)
    W = rand_bf16((9, 10), 13)
    ids = np.array([1, 8, 0, 4], dtype=np.int32)
    c = 3.5
    X2 = np.concatenate([X, f32_to_bf16_bits(np.ones((4, 1)))], axis=1)
    W2 = np.concatenate([W, f32_to_bf16_bits(np.full((9, 1), c))], axis=1)
    lp1, lz1 = oracle.logprobs(X, W, ids)
    lp2, lz2 = oracle.logprobs(X2, W2, ids)
    np.testing.assert_allclose(lp2, lp1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lz2, lz1 + c, rtol=0, atol=1e-12)


def test_dominant_logit():
    X = f32_to_bf16_bits(np.ones((1, 1)))
    W = f32_to_bf16_bits(np.array([[40.0], [0.0], [0.0], [0.0]]))
    for y, want in ((0, -math.log1p(3 * math.exp(-40.0))),
                    (2, -40.0 - math.log1p(3 * math.exp(-40.0)))):
        logp, logZ = oracle.logprobs(X, W, np.array([y], dtype=np.int32))
        assert logp[0] == pytest.approx(want, abs=1e-13)
    assert logZ[0] == pytest.approx(40.0, abs=1e-13)


def test_log_softmax_normalised_and_consistent():
    X = rand_bf16((6, 24), 14)
    W = rand_bf16((300, 24), 15, 0.5)
    ls = oracle.log_softmax(X, W)
    np.testing.assert_allclose(np.exp(ls).sum(axis=1), 1.0, rtol=0, atol=1e-12)
    ids = np.random.default_rng(16).integers(0, 300, 6).astype(np.int32)
    logp, _ = oracle.logprobs(X, W, ids)
    np.testing.assert_allclose(logp, ls[np.arange(6), ids], rtol=0, atol=1e-12)


def test_bad_id_gives_nan():
    X = rand_bf16((3, 8), 17)
    W = rand_bf16((5, 8), 18)
    logp, logZ = oracle.logprobs(X, W, np.array([-1, 5, 2], dtype=np.int32))
    assert math.isnan(logp[0]) and math.isnan(logp[1]) and not math.isnan(logp[2])
    assert np.all(np.isfinite(logZ))


# ----------------------------------------------------------------- leaves and tree
@pytest.mark.parametrize("n_leaves", [1, 2, 4, 8])
def test_leaf_sums_exact(n_leaves):
    H = 64
    x = rand_bf16((H,), 19)
    w = rand_bf16((H,), 20)
    got = oracle.leaf_sums(x, w, n_leaves)
    L = H // n_leaves
    xf = [bits_to_fraction(b) for b in x]
    wf = [bits_to_fraction(b) for b in w]
    for j in range(n_leaves):
        exact = sum(xf[k] * wf[k] for k in range(j * L, (j + 1) * L))
        assert got[j] == pytest.approx(float(exact), rel=1e-15, abs=1e-300)
    total = sum(xf[k] * wf[k] for k in range(H))
    assert math.fsum(got) == pytest.approx(float(total), rel=1e-14)


def _golden_tree(golden_dir):
    cases = []
    with open(os.path.join(golden_dir, "tree_fp32.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            n, ps, want, note = [s.strip() for s in line.split("|")]
            P = [float.fromhex(s) for s in ps.split()]
            assert len(P) == int(n)
            cases.append((int(n), P, float.fromhex(want), note))
    return cases


def test_tree_fp32_golden(golden_dir):
    cases = _golden_tree(golden_dir)
    assert len(cases) >= 6
    for n, P, want, note in cases:
        got = float(oracle.tree_fp32(np.array([P], dtype=np.float32))[0])
        assert got == want, (n, P, note)


def test_tree_fp32_rejects_non_power_of_two():
    assert math.isnan(float(oracle.tree_fp32(np.ones((1, 3), np.float32))[0]))


# ----------------------------------------------------------------- importance weights / D3
def _golden_is(golden_dir):
    rows, d3 = [], None
    with open(os.path.join(golden_dir, "importance_weights.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = [s.strip() for s in line.split("|")]
            if parts[0] == "D3":
                d3 = (float(parts[1]), int(parts[3]))
            else:
                rows.append(tuple(float(p) for p in parts))
    return rows, d3


def test_importance_weights_golden(golden_dir):
    rows, (d3_want, nv_want) = _golden_is(golden_dir)
    lp = np.array([r[0] for r in rows], np.float32)
    lm = np.array([r[1] for r in rows], np.float32)
    mask = np.array([int(r[2]) for r in rows], np.uint8)
    w, term, d3, nv = oracle.importance_weights(lp, lm, mask)
    for i, r in enumerate(rows):
        assert w[i] == pytest.approx(r[3], rel=1e-15)
        assert term[i] == pytest.approx(r[4], rel=1e-14, abs=1e-300)
    assert nv == nv_want
    assert d3 == pytest.approx(d3_want, rel=1e-15)


def test_d3_zero_when_weights_are_one():
    rng = np.random.default_rng(21)
    lp = rng.standard_normal(1000).astype(np.float32) * 3 - 5
    w, term, d3, nv = oracle.importance_weights(lp, lp.copy())
    assert np.all(w == 1.0) and np.all(term == 0.0)
    assert d3 == 0.0 and nv == 1000


def test_d3_small_gap_series():
    # e^d - 1 - d = d^2/2 + d^3/6 + d^4/24 + ...: the term must not lose digits near w = 1.
    d = np.array([1e-3, -1e-3, 2.0 ** -12, -(2.0 ** -20)], np.float32)
    w, term, _, _ = oracle.importance_weights(d, np.zeros_like(d))
    for di, ti in zip(d.astype(np.float64), term):
        series = di * di / 2 + di ** 3 / 6 + di ** 4 / 24 + di ** 5 / 120
        assert ti == pytest.approx(series, rel=1e-12)


def test_d3_mask_and_empty():
    lp = np.array([0.5, -1.0], np.float32)
    lm = np.zeros(2, np.float32)
    _, _, d3, nv = oracle.importance_weights(lp, lm, np.zeros(2, np.uint8))
    assert d3 == 0.0 and nv == 0
    _, _, d3, nv = oracle.importance_weights(np.zeros(0, np.float32), np.zeros(0, np.float32))
    assert d3 == 0.0 and nv == 0


def test_term_nonnegative_and_w_positive():
    rng = np.random.default_rng(22)
    lp = rng.uniform(-20, 0, 5000).astype(np.float32)
    lm = rng.uniform(-20, 0, 5000).astype(np.float32)
    w, term, d3, nv = oracle.importance_weights(lp, lm)
    assert np.all(w > 0) and np.all(term >= 0) and d3 > 0 and nv == 5000


# ----------------------------------------------------------------- acceptance statistics
def test_acceptance_stats_identical_inputs_all_zero():
    rng = np.random.default_rng(30)
    a = rng.uniform(-30, 0, 4000).astype(np.float32)
    st = oracle.acceptance_stats(a, a.copy())
    assert (st["max"], st["mean"], st["std"], st["k3"], st["n_valid"]) == (0.0, 0.0, 0.0, 0.0, 4000)


def test_acceptance_stats_constant_gap_closed_form():
    # a - b = 1/2 exactly on every token (b on a 1/8 grid): max = mean = 1/2, std = 0,
    # k3 = e^(1/2) - 1 - 1/2.
    b = (-np.arange(0, 640) / 8.0).astype(np.float32)
    a = (b + 0.5).astype(np.float32)
    st = oracle.acceptance_stats(a, b)
    assert st["max"] == 0.5 and st["mean"] == 0.5 and st["std"] == 0.0
    # (640 equal terms summed in fp64: relative error below 640 * 2^-53)
    assert abs(st["k3"] - (math.exp(0.5) - 1.5)) < 1e-13 * st["k3"]
    st = oracle.acceptance_stats(b, a)  # r = e^(-1/2)
    assert abs(st["k3"] - (math.exp(-0.5) - 1 + 0.5)) < 1e-13 * st["k3"]


def test_acceptance_stats_against_library_statistics():
    import statistics

    rng = np.random.default_rng(31)
    a = rng.uniform(-12, 0, 3001).astype(np.float32)
    b = (a + rng.normal(0, 0.05, a.size)).astype(np.float32)
    mask = rng.random(a.size) < 0.7
    st = oracle.acceptance_stats(a, b, mask)
    gaps = [abs(Fraction(float(x)) - Fraction(float(y))) for x, y, m in zip(a, b, mask) if m]
    assert st["n_valid"] == len(gaps)
    assert st["max"] == float(max(gaps))
    assert abs(st["mean"] - float(statistics.fmean(gaps))) < 1e-15
    assert abs(st["std"] - statistics.pstdev([float(g) for g in gaps])) < 1e-14
    # k3 is the D3 term on the same tokens
    _, _, d3, nv = oracle.importance_weights(a, b, mask)
    assert nv == st["n_valid"] and abs(st["k3"] - d3) < 1e-15


def test_acceptance_stats_nan_mask_and_empty():
    a = np.array([0.0, -1.0, np.nan, -2.0], dtype=np.float32)
    b = np.array([0.0, -1.5, -3.0, -2.0], dtype=np.float32)
    st = oracle.acceptance_stats(a, b, [1, 1, 0, 1])  # NaN token masked out
    assert st["max"] == 0.5 and st["n_valid"] == 3
    st = oracle.acceptance_stats(a, b)
    assert all(math.isnan(st[k]) for k in ("max", "mean", "std", "k3"))
    st = oracle.acceptance_stats(a, b, [0, 0, 0, 0])
    assert st == dict(max=0.0, mean=0.0, std=0.0, k3=0.0, n_valid=0)


# ----------------------------------------------------------------- REINFORCE Zero loss
def test_reinforce_zero_worked_example():
    # Two groups of two responses; rewards (1, 0 | 1/2, 1/2) give A = (1/2, -1/2, 0, 0).
    # Response 0: tokens with w = 2 and 1 (mean 3/2); response 1: one token with w = 4.
    # L = -(1/4) (1/2 * 3/2 - 1/2 * 4) = 5/16.  dL/dlog pi = -(1/4)(1/T_i) A_i w:
    # -1/8, -1/16 | 1/2 | 0 0 0 | 0.
    lp = np.array([math.log(2), 0, math.log(4), 0, 0, 0, 0], dtype=np.float32)
    out = oracle.reinforce_zero(lp, np.zeros(7, np.float32), [0, 2, 3, 6, 7],
                                [1, 0, 0.5, 0.5], 2)
    assert abs(out["loss"] - 5 / 16) < 1e-6
    assert np.allclose(out["grad"], [-1 / 8, -1 / 16, 1 / 2, 0, 0, 0, 0], rtol=1e-6, atol=0)
    assert np.array_equal(out["adv"], [0.5, -0.5, 0.0, 0.0])
    # masking response 0's second token makes its token mean 2: L = -(1/4)(1 - 2) = 1/4
    out = oracle.reinforce_zero(lp, np.zeros(7, np.float32), [0, 2, 3, 6, 7],
                                [1, 0, 0.5, 0.5], 2, mask=[1, 0, 1, 1, 1, 1, 1])
    assert abs(out["loss"] - 1 / 4) < 1e-6 and out["grad"][1] == 0.0 and out["w_hat"][1] == 0.0


def _rz_case(seed, B=8, G=4, lag=0.05):
    rng = np.random.default_rng(seed)
    lens = rng.integers(1, 40, B)
    offs = np.concatenate([[0], np.cumsum(lens)])
    T = int(offs[-1])
    # logprobs on a 2^-10 grid so that +-2^-12 perturbations are exact in fp32
    lm = (np.round(rng.uniform(-6, -0.1, T) * 1024) / 1024).astype(np.float32)
    lp = (lm + np.round(rng.normal(0, lag, T) * 1024) / 1024).astype(np.float32)
    rewards = rng.integers(0, 2, B).astype(np.float32)
    mask = rng.random(T) < 0.85
    return lp, lm, offs, rewards, G, mask


def test_reinforce_zero_equal_policies_give_zero_loss():
    # w = 1 everywhere: L = -(1/B) sum_i A_i, and group-centred advantages sum to 0
    lp, lm, offs, rewards, G, mask = _rz_case(40)
    mask[offs[:-1]] = True  # every response keeps a valid token
    out = oracle.reinforce_zero(lp, lp, offs, rewards, G, mask=mask)
    assert abs(out["loss"]) < 1e-15
    assert np.all(out["w_hat"][mask] == 1.0)


@pytest.mark.parametrize("opts", [
    dict(),
    dict(flags=oracle.TIS, tis_cap=1.03),
    dict(flags=oracle.TOKEN_GATE, token_log_lo=-0.06, token_log_hi=0.06),
    dict(flags=oracle.SEQ_GATE, seq_log_lo=-0.3, seq_log_hi=0.3),
], ids=["plain", "tis", "token_gate", "seq_gate"])
def test_reinforce_zero_gradient_is_the_derivative_of_the_loss(opts):
    lp, lm, offs, rewards, G, mask = _rz_case(41)
    out = oracle.reinforce_zero(lp, lm, offs, rewards, G, mask=mask, **opts)
    h = 2.0 ** -12
    d = lp.astype(np.float64) - lm
    checked = 0
    for t in range(lp.size):
        w = math.exp(d[t])
        # stay inside one smooth piece: away from the cap and the gate edges
        if "tis_cap" in opts and abs(w - opts["tis_cap"]) < 4 * h * w:
            continue
        if "token_log_lo" in opts and min(abs(d[t] - 0.06), abs(d[t] + 0.06)) < 2 * h:
            continue
        i = np.searchsorted(offs, t, side="right") - 1
        if "seq_log_lo" in opts and min(abs(out["seq_logratio"][i] - 0.3),
                                        abs(out["seq_logratio"][i] + 0.3)) < 2 * h:
            continue
        up, dn = lp.copy(), lp.copy()
        up[t] += np.float32(h)
        dn[t] -= np.float32(h)
        lu = oracle.reinforce_zero(up, lm, offs, rewards, G, mask=mask, **opts)["loss"]
        ld = oracle.reinforce_zero(dn, lm, offs, rewards, G, mask=mask, **opts)["loss"]
        fd = (lu - ld) / (2 * h)
        g = out["grad"][t]
        if opts.get("flags", 0) & (oracle.TIS | oracle.TOKEN_GATE | oracle.SEQ_GATE):
            # the modified weight is a coefficient of grad log pi: d/dlog pi of w_hat is
            # w_hat where it tracks w, 0 where it is capped or gated
            capped = "tis_cap" in opts and w > opts["tis_cap"]
            if capped:
                assert abs(fd) < 1e-9, (t, fd)
                assert abs(g - out["grad"][t]) == 0.0
                checked += 1
                continue
        assert abs(fd - g) <= 1e-6 * max(abs(g), 1e-3), (t, fd, g)
        checked += 1
    assert checked > lp.size // 2


def test_reinforce_zero_tis_and_gate_limits():
    lp, lm, offs, rewards, G, mask = _rz_case(42)
    plain = oracle.reinforce_zero(lp, lm, offs, rewards, G, mask=mask)
    big = oracle.reinforce_zero(lp, lm, offs, rewards, G, mask=mask, flags=oracle.TIS,
                                tis_cap=1e30)
    assert big["loss"] == plain["loss"] and np.array_equal(big["grad"], plain["grad"])
    open_gates = oracle.reinforce_zero(lp, lm, offs, rewards, G, mask=mask,
                                       flags=oracle.TOKEN_GATE | oracle.SEQ_GATE)
    assert open_gates["loss"] == plain["loss"] and open_gates["kept"].all()
    # a cap below every weight makes w_hat constant, so the centred advantages cancel
    mask[offs[:-1]] = True
    tiny = oracle.reinforce_zero(lp, lm, offs, rewards, G, mask=mask, flags=oracle.TIS,
                                 tis_cap=1e-3)
    assert np.all(tiny["w_hat"][mask] == 1e-3) and abs(tiny["loss"]) < 1e-15


def test_reinforce_zero_sequence_gate_drops_whole_responses():
    # response 0: four tokens with d = 1/4 (log-ratio 1); response 1: d = 1/8 twice (1/4)
    lm = np.full(8, -2.0, dtype=np.float32)
    lp = lm + np.array([0.25] * 4 + [0.125] * 2 + [0, 0], dtype=np.float32)
    offs, rewards = [0, 4, 6, 7, 8], [1, 0, 1, 0]
    out = oracle.reinforce_zero(lp, lm, offs, rewards, 2, flags=oracle.SEQ_GATE,
                                seq_log_lo=-0.9, seq_log_hi=0.9)
    assert out["kept"].tolist() == [False, True, True, True]
    assert out["seq_logratio"][0] == 1.0 and out["seq_logratio"][1] == 0.25
    assert np.all(out["w_hat"][:4] == 0) and np.all(out["grad"][:4] == 0)
    # the same as a plain loss with response 0 masked out (T_0 = 0 adds nothing)
    masked = oracle.reinforce_zero(lp, lm, offs, rewards, 2, mask=[0] * 4 + [1] * 4)
    assert out["loss"] == masked["loss"]
    assert abs(out["loss"] - (-(1 / 4) * (-0.5 * math.exp(0.125) + 0.5 - 0.5))) < 1e-7


def test_reinforce_zero_token_gate_and_empty_response():
    lm = np.full(6, -1.0, dtype=np.float32)
    lp = lm + np.array([0.5, 0.0, -0.5, 0.0, 0.0, 0.0], dtype=np.float32)
    out = oracle.reinforce_zero(lp, lm, [0, 3, 3, 6, 6], [1, 0, 0, 1], 2,
                                flags=oracle.TOKEN_GATE, token_log_lo=-0.25, token_log_hi=0.25)
    assert out["w_hat"].tolist() == [0.0, 1.0, 0.0, 1.0, 1.0, 1.0]
    # responses 1 and 3 are empty: they add nothing and give no NaN
    assert np.isfinite(out["loss"]) and np.isfinite(out["grad"]).all()
    assert abs(out["loss"] - (-(1 / 4) * (0.5 * (1 / 3) - 0.5 * 1.0))) < 1e-15


# ----------------------------------------------------------------- entropy
def test_entropy_closed_forms():
    # uniform logits: log V; two tokens: the binary entropy of sigmoid(z_1 - z_0)
    V, H = 1000, 16
    X = rand_bf16((3, H), 50)
    W = np.repeat(rand_bf16((1, H), 51), V, axis=0)
    np.testing.assert_allclose(oracle.entropy(X, W), math.log(V), rtol=0, atol=1e-12)
    X = rand_bf16((5, 6), 52)
    W = rand_bf16((2, 6), 53, 2.0)
    ex = exact_logits(X, W)
    ent = oracle.entropy(X, W)
    for t in range(5):
        p = 1.0 / (1.0 + math.exp(float(ex[t][0] - ex[t][1])))
        want = -(p * math.log(p) + (1 - p) * math.log1p(-p))
        assert ent[t] == pytest.approx(want, abs=1e-13)


def test_entropy_bounds_and_decimal_brute_force():
    X = rand_bf16((3, 8), 54)
    W = rand_bf16((11, 8), 55, 3.0)
    ent = oracle.entropy(X, W)
    ex = exact_logits(X, W)
    for t in range(3):
        zs = [dec(z) for z in ex[t]]
        total = sum((z.exp() for z in zs), Decimal(0))
        lz = total.ln()
        want = -sum(((z - lz).exp() * (z - lz) for z in zs), Decimal(0))
        assert ent[t] == pytest.approx(float(want), abs=1e-14)
        assert 0.0 <= ent[t] <= math.log(11) + 1e-15
    # one dominant logit: the entropy vanishes like 40 * 3 e^-40
    X1 = f32_to_bf16_bits(np.ones((1, 1)))
    W1 = f32_to_bf16_bits(np.array([[40.0], [0.0], [0.0], [0.0]]))
    assert oracle.entropy(X1, W1)[0] == pytest.approx(41 * 3 * math.exp(-40.0), rel=1e-6)


# ----------------------------------------------------------------- logprob gradient
def test_logprobs_f64_matches_the_bf16_path():
    X = rand_bf16((6, 24), 56)
    W = rand_bf16((37, 24), 57)
    ids = np.random.default_rng(58).integers(0, 37, 6).astype(np.int32)
    lp, _ = oracle.logprobs(X, W, ids)
    Xd = np.array([[float(bits_to_fraction(b)) for b in row] for row in X])
    Wd = np.array([[float(bits_to_fraction(b)) for b in row] for row in W])
    np.testing.assert_allclose(oracle.logprobs_f64(Xd, Wd, ids), lp, rtol=0, atol=1e-13)


def test_logprob_grad_is_the_derivative():
    T, H, V = 3, 5, 7
    X = rand_bf16((T, H), 59)
    W = rand_bf16((V, H), 60, 1.5)
    ids = np.array([0, 6, 3], dtype=np.int32)
    g = np.array([0.7, -1.3, 2.0])
    dX, dW, dl = oracle.logprob_grad(X, W, ids, g)
    Xd = np.array([[float(bits_to_fraction(b)) for b in row] for row in X])
    Wd = np.array([[float(bits_to_fraction(b)) for b in row] for row in W])
    L = lambda Xv, Wv: float(np.dot(g, oracle.logprobs_f64(Xv, Wv, ids)))  # noqa: E731
    h = 1e-6
    for t in range(T):
        for k in range(H):
            up, dn = Xd.copy(), Xd.copy()
            up[t, k] += h
            dn[t, k] -= h
            assert (L(up, Wd) - L(dn, Wd)) / (2 * h) == pytest.approx(dX[t, k], abs=1e-8)
    for v in range(V):
        for k in range(H):
            up, dn = Wd.copy(), Wd.copy()
            up[v, k] += h
            dn[v, k] -= h
            assert (L(Xd, up) - L(Xd, dn)) / (2 * h) == pytest.approx(dW[v, k], abs=1e-8)
    # each row of dl sums to 0 (probabilities sum to 1), so the columns of dW sum to 0
    np.testing.assert_allclose(dl.sum(axis=1), 0.0, atol=1e-14)
    np.testing.assert_allclose(dW.sum(axis=0), 0.0, atol=1e-13)


def test_logprob_grad_identical_rows_give_zero_dx():
    V, H = 64, 12
    X = rand_bf16((4, H), 61)
    W = np.repeat(rand_bf16((1, H), 62), V, axis=0)
    dX, _, dl = oracle.logprob_grad(X, W, np.array([3, 0, 63, 9], dtype=np.int32), np.ones(4))
    np.testing.assert_allclose(dX, 0.0, atol=1e-14)
    np.testing.assert_allclose(dl[0, 3], 1 - 1 / V, rtol=1e-14)


# ----------------------------------------------------------------- block FP8
def _torch_e4m3():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("this torch has no float8_e4m3fn")
    return torch


def test_e4m3_codes_match_the_library_format():
    torch = _torch_e4m3()
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().double().numpy()
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.array_equal(ours[~np.isnan(ours)], ref[~np.isnan(ref)])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def test_e4m3_rounding_matches_the_library_and_saturates():
    torch = _torch_e4m3()
    rng = np.random.default_rng(70)
    x = np.concatenate([rng.uniform(-448, 448, 20000), rng.uniform(-0.03, 0.03, 20000),
                        # exact ties between neighbours: 1 + 1/16 lies between 1 and 1.125
                        [1.0625, -1.0625, 1.1875, 2.0 ** -10, 3 * 2.0 ** -10, 416.0, 432.0]])
    x = x.astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.e4m3_encode(x), ref)
    assert oracle.e4m3_encode([1.0625])[0] == 0x38          # tie to the even mantissa: 1.0
    assert oracle.e4m3_encode([1.1875])[0] == 0x3A          # tie to even: 1.25
    sat = oracle.e4m3_encode([449.0, 1e30, -500.0, 464.0])
    assert sat.tolist() == [0x7E, 0x7E, 0xFE, 0x7E]         # saturate to +-448


def test_block_quantisation_rule():
    rng = np.random.default_rng(71)
    M = f32_to_bf16_bits(rng.standard_normal((130, 256)).astype(np.float32) * 0.05)
    M[7, 3:131] = 0  # an all-zero 1 x 128 block
    for block_rows in (1, 128):
        q, s = oracle.quantize_blocks(M, block_rows)
        vals = np.array([[float(bits_to_fraction(b)) for b in row] for row in M], dtype=np.float32)
        for rb in range(s.shape[0]):
            for kb in range(2):
                blk = vals[rb * block_rows:(rb + 1) * block_rows, kb * 128:(kb + 1) * 128]
                amax = np.float32(np.abs(blk).max())
                want = np.float32(amax / np.float32(448.0)) if amax > 0 else np.float32(1.0)
                assert s[rb, kb] == want
                deq = oracle.e4m3_decode(q[rb * block_rows:(rb + 1) * block_rows,
                                           kb * 128:(kb + 1) * 128]).reshape(blk.shape)
                if amax > 0:
                    assert np.abs(deq).max() == 448.0  # the block maximum maps to +-448
                # every value within half a step of its e4m3 neighbour (relative 2^-4)
                err = np.abs(deq - blk.astype(np.float64) / float(s[rb, kb]))
                assert np.all(err <= np.maximum(np.abs(deq) * 2.0 ** -4, 2.0 ** -10))


def test_logprobs_fp8_equals_the_bf16_oracle_on_representable_inputs():
    # blocks whose maximum is 448 and whose values are e4m3 numbers quantise to themselves
    # with scale 1, so the block-FP8 logprob must equal the bf16 logprob of the same values
    rng = np.random.default_rng(72)
    grid = oracle.e4m3_decode(np.arange(1, 0x7F, dtype=np.uint8))  # nonzero, so signs survive
    grid = np.concatenate([grid, -grid])
    def rep(shape):
        v = rng.choice(grid[np.abs(grid) <= 2.0], size=shape)
        v[:, ::128] = 448.0
        return v.astype(np.float32)
    X = f32_to_bf16_bits(rep((5, 256)) / 1.0)
    W = f32_to_bf16_bits(np.concatenate([rep((128, 256)), rep((3, 256))]))
    ids = np.array([0, 130, 7, 64, 129], dtype=np.int32)
    xq, sx = oracle.quantize_blocks(X, 1)
    wq, sw = oracle.quantize_blocks(W, 128)
    assert np.all(sx == 1.0) and np.all(sw == 1.0)
    lp8, lz8 = oracle.logprobs_fp8(xq, sx, wq, sw, ids)
    lp, lz = oracle.logprobs(X, W, ids)
    np.testing.assert_allclose(lp8, lp, rtol=0, atol=1e-9)
    np.testing.assert_allclose(lz8, lz, rtol=1e-15, atol=0)
    # and scaling a weight block by 2^-3 moves its scale, not its codes
    W2 = W.copy()
    W2[:128, 128:] = f32_to_bf16_bits(np.array([[float(bits_to_fraction(b)) for b in row]
                                                 for row in W[:128, 128:]]) / 8.0)
    wq2, sw2 = oracle.quantize_blocks(W2, 128)
    assert np.array_equal(wq2, wq) and sw2[0, 1] == 0.125 and sw2[0, 0] == 1.0
    # with unequal (power-of-two) block scales the dequantised values are still exact in bf16
    lp8, lz8 = oracle.logprobs_fp8(xq, sx, wq2, sw2, ids)
    lp, lz = oracle.logprobs(X, W2, ids)
    np.testing.assert_allclose(lp8, lp, rtol=0, atol=1e-9)
    np.testing.assert_allclose(lz8, lz, rtol=1e-15, atol=0)


def test_entropy_fp8_equals_the_bf16_oracle_on_representable_inputs():
    # the same representable blocks as above: the block-FP8 entropy must equal the (pinned)
    # bf16 entropy of the same values, with unit scales and with a weight block at 2^-3
    rng = np.random.default_rng(73)
    grid = oracle.e4m3_decode(np.arange(1, 0x7F, dtype=np.uint8))
    grid = np.concatenate([grid, -grid])
    def rep(shape):
        v = rng.choice(grid[np.abs(grid) <= 2.0], size=shape)
        v[:, ::128] = 448.0
        return v.astype(np.float32)
    X = f32_to_bf16_bits(rep((4, 256)) / 64.0)   # power-of-two activation scales (7/64)
    W = f32_to_bf16_bits(np.concatenate([rep((128, 256)), rep((5, 256))]) / 256.0)
    W[:128, 128:] = f32_to_bf16_bits(np.array([[float(bits_to_fraction(b)) for b in row]
                                                for row in W[:128, 128:]]) / 8.0)
    xq, sx = oracle.quantize_blocks(X, 1)
    wq, sw = oracle.quantize_blocks(W, 128)
    assert len(set(sw.ravel().tolist())) == 2 and np.all(sx == sx.ravel()[0])
    np.testing.assert_allclose(oracle.entropy_fp8(xq, sx, wq, sw), oracle.entropy(X, W),
                               rtol=1e-13, atol=1e-12)
    # rows subset, in the order given
    np.testing.assert_allclose(oracle.entropy_fp8(xq, sx, wq, sw, rows=[3, 0]),
                               oracle.entropy(X, W, rows=[3, 0]), rtol=1e-13, atol=1e-12)


def test_fp8_activation_scales_indexed_by_row_and_block():
    # Activation blocks (1 x 128, one scale per row and per 128-K block; the DeepSeek block
    # rule the vLLM blog keeps for block-FP8) whose scales are unequal powers of two that
    # differ along the row AND along K.  Each block holds e4m3 grid values times its scale, so
    # it quantises to the grid codes with exactly that scale, and the dequantised operands are
    # the bf16 values themselves: the block-FP8 logprob and entropy must equal the (pinned)
    # bf16 oracle's.  A scale read from another row or another block changes the logits.
    rng = np.random.default_rng(75)
    grid = oracle.e4m3_decode(np.arange(1, 0x7F, dtype=np.uint8))
    grid = np.concatenate([grid, -grid])
    def rep(shape):
        v = rng.choice(grid[np.abs(grid) <= 2.0], size=shape)
        v[:, ::128] = 448.0
        return v.astype(np.float32)
    expo = np.array([[0, 3], [2, 1], [5, 0], [1, 4], [3, 2]])  # 2^-e per (row, K block)
    xv = rep((5, 256))
    for r in range(5):
        for kb in range(2):
            xv[r, kb * 128:(kb + 1) * 128] /= np.float32(2.0 ** expo[r, kb])
    X = f32_to_bf16_bits(xv)
    W = f32_to_bf16_bits(np.concatenate([rep((128, 256)), rep((6, 256))]) / 16.0)
    ids = np.array([3, 131, 64, 0, 100], dtype=np.int32)
    xq, sx = oracle.quantize_blocks(X, 1)
    wq, sw = oracle.quantize_blocks(W, 128)
    assert sx.shape == (5, 2)
    np.testing.assert_array_equal(sx, (2.0 ** -expo).astype(np.float32))
    assert len(set(sx[:, 0].tolist())) > 1 and np.any(sx[:, 0] != sx[:, 1])
    lp8, lz8 = oracle.logprobs_fp8(xq, sx, wq, sw, ids)
    lp, lz = oracle.logprobs(X, W, ids)
    np.testing.assert_allclose(lp8, lp, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lz8, lz, rtol=1e-15, atol=1e-15)
    assert np.ptp(lp) > 0.1  # the logits really vary between tokens
    np.testing.assert_allclose(oracle.entropy_fp8(xq, sx, wq, sw), oracle.entropy(X, W),
                               rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(oracle.entropy_fp8(xq, sx, wq, sw, rows=[4, 1]),
                               oracle.entropy(X, W, rows=[4, 1]), rtol=1e-13, atol=1e-13)


def test_entropy_fp8_of_a_zero_lm_head_is_log_v():
    X = f32_to_bf16_bits(np.random.default_rng(74).standard_normal((3, 128)).astype(np.float32))
    W = np.zeros((300, 128), dtype=np.uint16)
    xq, sx = oracle.quantize_blocks(X, 1)
    wq, sw = oracle.quantize_blocks(W, 128)
    np.testing.assert_allclose(oracle.entropy_fp8(xq, sx, wq, sw), np.log(300.0), rtol=1e-14)


# ----------------------------------------------------------------- planted mistakes
MUTATIONS = [
    # (description, original text, mutated text)
    ("sign of the logprob", "? z[y] - lz : NAN", "? lz - z[y] : NAN"),
    ("log-sum-exp without the max term", "return m + log(s);", "return log(s);"),
    ("transposed row index", "z[r * V + v] = logit_f64(xrow, W + v * H, H);",
     "z[r * V + v] = logit_f64(X + v * ldx, W + rows[r] * H, H);"),
    ("interleaved tree pairing", "buf[i] = a + b;", "buf[i] = buf[i] + buf[i + n / 2];"),
    ("ratio inverted", "double d = (double)logp_pi[t] - (double)logp_mu[t];",
     "double d = (double)logp_mu[t] - (double)logp_pi[t];"),
    ("term drops the -d", "term[t] = expm1(d) - d;", "term[t] = expm1(d);"),
    ("leaf boundary off by one", "k < (int64_t)(j + 1) * L; ++k", "k <= (int64_t)(j + 1) * L && k < H; ++k"),
    ("std with n - 1", "out[2] = sqrt(ss / (double)n);", "out[2] = sqrt(ss / (double)(n - 1));"),
    ("k3 drops the -d", "k3 += expm1(d) - d;", "k3 += expm1(d);"),
    ("advantage not centred", "double A = (double)rewards[i] - gsum / (double)G;",
     "double A = (double)rewards[i];"),
    ("groups strided", "int64_t g0 = (i / G) * G;", "int64_t g0 = (i % G) * G;"),
    ("token mean over masked tokens too", "if (n > 0) total += A * wsum / (double)n;",
     "if (n > 0) total += A * wsum / (double)(offs[i + 1] - offs[i]);"),
    ("gradient sign", "double coef = n > 0 ? -A /", "double coef = n > 0 ? A /"),
    ("TIS as a floor", "wh > tis_cap) wh = tis_cap;", "wh < tis_cap) wh = tis_cap;"),
    ("entropy sign", "if (p > 0.0) h -= p * lp;", "if (p > 0.0) h += p * lp;"),
    ("FP8 entropy sign", "if (pv > 0.0) h -= pv * lpv;", "if (pv > 0.0) h += pv * lpv;"),
    ("FP8 entropy with the activation scale for the weights",
     "acc += xd[k] * (oracle_e4m3_decode(wrow[k]) * (double)swrow[k / 128]);",
     "acc += xd[k] * (oracle_e4m3_decode(wrow[k]) * (double)sxrow[k / 128]);"),
    ("gradient without the one-hot term", "dl[t * V + v] = g[t] * (onehot - exp(z[v] - lz));",
     "dl[t * V + v] = g[t] * (-exp(z[v] - lz));"),
    ("gradient with unnormalised probabilities", "dl[t * V + v] = g[t] * (onehot - exp(z[v] - lz));",
     "dl[t * V + v] = g[t] * (onehot - exp(z[v]));"),
    ("dW with a transposed operand", "acc += dl[t * V + v] * bf16_to_f64(X[t * H + k]);",
     "acc += dl[t * V + v] * bf16_to_f64(W[v * H + k]);"),
    ("e4m3 ties away from zero", "double m = nearbyint((a / ldexp(1.0, e) - 1.0) * 8.0);",
     "double m = floor((a / ldexp(1.0, e) - 1.0) * 8.0 + 0.5);"),
    ("e4m3 without saturation", "if (a >= 448.0) return sgn | 0x7E;", "if (a >= 480.0) return sgn | 0x7F;"),
    ("block scale against 224", "float s = amax > 0.0f ? amax / 448.0f : 1.0f;",
     "float s = amax > 0.0f ? amax / 224.0f : 1.0f;"),
    ("weight scale with a transposed block index", "(double)sw[(v / 128) * nkb + k / 128]",
     "(double)sw[(k / 128) * nkb + v / 128]"),
    ("FP8 activation scale without the row index",
     "(double)sx[t * nkb + k / 128];", "(double)sx[k / 128];"),
    ("FP8 activation scale without the block index",
     "(double)sx[t * nkb + k / 128];", "(double)sx[t * nkb];"),
    ("FP8 entropy activation scale without the row index",
     "const float* sxrow = sx + t * nkb;", "const float* sxrow = sx;"),
    ("FP8 entropy activation scale without the block index",
     "xd[k] = oracle_e4m3_decode(xq[t * H + k]) * (double)sxrow[k / 128];",
     "xd[k] = oracle_e4m3_decode(xq[t * H + k]) * (double)sxrow[0];"),
    ("sequence gate on the last token only", "lr += (double)logp_pi[t] - (double)logp_mu[t];",
     "lr = (double)logp_pi[t] - (double)logp_mu[t];"),
]


def _build_mutant(tmp_path, original, mutated):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    assert original in src, original
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(original, mutated))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                           "-std=c11", "-o", str(lib), str(path), "-lm"])
    return str(lib)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("desc,original,mutated", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, monkeypatch, golden_dir, desc, original, mutated):
    """Swap the oracle library for a mutated build; at least one pin above must fail."""
    lib_path = _build_mutant(tmp_path, original, mutated)
    monkeypatch.setattr(oracle, "_lib", None)
    monkeypatch.setattr(oracle, "build", lambda force=False: lib_path)
    pins = [test_logits_exact_rational, test_logits_rows_subset_and_orientation,
            test_logprobs_brute_force_decimal, test_two_token_vocab_closed_form,
            test_uniform_logits_give_minus_log_v, test_dominant_logit,
            lambda: test_tree_fp32_golden(golden_dir),
            lambda: test_importance_weights_golden(golden_dir),
            lambda: [test_leaf_sums_exact(n) for n in (2, 4, 8)],
            test_d3_small_gap_series,
            test_acceptance_stats_constant_gap_closed_form,
            test_acceptance_stats_against_library_statistics,
            test_reinforce_zero_worked_example,
            test_reinforce_zero_equal_policies_give_zero_loss,
            lambda: [test_reinforce_zero_gradient_is_the_derivative_of_the_loss(o) for o in (
                dict(), dict(flags=oracle.TIS, tis_cap=1.03))],
            test_reinforce_zero_tis_and_gate_limits,
            test_reinforce_zero_sequence_gate_drops_whole_responses,
            test_reinforce_zero_token_gate_and_empty_response,
            test_entropy_closed_forms, test_entropy_bounds_and_decimal_brute_force,
            test_logprob_grad_is_the_derivative, test_logprob_grad_identical_rows_give_zero_dx,
            test_e4m3_codes_match_the_library_format,
            test_e4m3_rounding_matches_the_library_and_saturates, test_block_quantisation_rule,
            test_logprobs_fp8_equals_the_bf16_oracle_on_representable_inputs,
            test_entropy_fp8_equals_the_bf16_oracle_on_representable_inputs,
            test_entropy_fp8_of_a_zero_lm_head_is_log_v,
            test_fp8_activation_scales_indexed_by_row_and_block]
    failed = 0
    for pin in pins:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            failed += 1
    monkeypatch.setattr(oracle, "_lib", None)
    assert failed > 0, f"no pin caught the planted mistake: {desc}"
