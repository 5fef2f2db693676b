"""GPU parity against the fp64 CPU oracle, through the C ABI, on small shapes that still
span several tiles and a ragged tail.

Tolerances: the engine must match the oracle within 2e-3 nats (the contract).  The
arithmetic itself bounds the error far lower -- fp32 leaf sums over at most a few
hundred products, a tree of at most 3 adds, and fp32 exp/log over <= 1187 tiles -- so
the tests also assert a derived 1e-4 bound, to catch mistakes that stay inside 2e-3.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from bit_consistent_logprob_gb300 import Engine, LpError, inputs
from bit_consistent_logprob_gb300.inputs import WORKLOADS

from gpu_util import LOGP_TOL, assert_bit_equal, bits, require_cuda

pytestmark = pytest.mark.gpu
DERIVED_TOL = 1e-4


@pytest.fixture(scope="module")
def dev():
    return require_cuda()


@pytest.fixture(scope="module")
def tiny(dev):
    wl = WORKLOADS["tiny"]
    X = inputs.hidden_states(wl.T, wl.H, wl.seed)
    W = inputs.lm_head(wl.V, wl.H, wl.seed)
    ls = oracle.log_softmax(X, W)
    ids = inputs.gumbel_max_ids(ls, wl.seed)
    return wl, X, W, ids, ls


def run(W, X, ids, n_leaves, dev, tp_slices=1, max_tokens=None, phase=0):
    with Engine(W.to(dev), n_leaves=n_leaves, tp_slices=tp_slices,
                max_tokens=max_tokens or max(1, X.shape[0])) as eng:
        logp, logZ = eng.logprobs(X.to(dev), ids.to(dev), return_logZ=True, phase=phase)
        eng.check()
    return logp, logZ


def test_tiny_logprobs_match_oracle(tiny, dev):
    wl, X, W, ids, ls = tiny
    logp, logZ = run(W, X, ids, wl.n_leaves, dev)
    rows = np.arange(wl.T)
    want = ls[rows, ids.numpy()]
    err = np.abs(logp.cpu().double().numpy() - want)
    assert err.max() <= LOGP_TOL
    assert err.max() <= DERIVED_TOL, err.max()
    _, lz_ref = oracle.logprobs(X, W, ids.numpy())
    assert np.abs(logZ.cpu().double().numpy() - lz_ref).max() <= DERIVED_TOL


def test_leaf_partials_within_fp32_bound(tiny, dev):
    # Each exported leaf partial is an fp32 accumulation of L = H/N products: it must lie
    # within a few units of L * 2^-24 * sum|x w| of the exact leaf sum.
    wl, X, W, ids, _ = tiny
    N, L = wl.n_leaves, wl.H // wl.n_leaves
    with Engine(W.to(dev), n_leaves=N, max_tokens=wl.T) as eng:
        parts = [eng.logits_partial(X.to(dev), j, 1).cpu() for j in range(N)]
        eng.check()
    rng = np.random.default_rng(3)
    xs, ws = X.float().numpy().astype(np.float64), W.float().numpy().astype(np.float64)
    for _ in range(200):
        t, v = int(rng.integers(wl.T)), int(rng.integers(wl.V))
        exact = oracle.leaf_sums(X[t], W[v], N)
        for j in range(N):
            k = slice(j * L, (j + 1) * L)
            mag = np.abs(xs[t, k] * ws[v, k]).sum()
            bound = 4 * L * 2.0 ** -24 * mag + 1e-30
            assert abs(float(parts[j][t, v]) - exact[j]) <= bound, (t, v, j)


def test_leaf_tree_is_bit_exact(tiny, dev):
    # The full tree node equals the oracle's fp32 pairwise tree over the exported leaves.
    wl, X, W, _, _ = tiny
    N = wl.n_leaves
    with Engine(W.to(dev), n_leaves=N, max_tokens=wl.T) as eng:
        Xd = X.to(dev)
        parts = torch.stack([eng.logits_partial(Xd, j, 1).cpu() for j in range(N)], dim=-1)
        full = eng.logits_partial(Xd, 0, N).cpu()
        half0 = eng.logits_partial(Xd, 0, N // 2).cpu()
        eng.check()
    want = torch.from_numpy(oracle.tree_fp32(parts.numpy()))
    assert_bit_equal(full, want, "full tree node vs oracle fp32 tree")
    want_half = torch.from_numpy(oracle.tree_fp32(parts[..., : N // 2].numpy()))
    assert_bit_equal(half0, want_half, "left subtree vs oracle fp32 tree")


@pytest.mark.parametrize("s", [2, 4])
def test_tp_split_is_bit_identical(tiny, dev, s):
    wl, X, W, ids, _ = tiny
    base, baseZ = run(W, X, ids, wl.n_leaves, dev)
    tp, tpZ = run(W, X, ids, wl.n_leaves, dev, tp_slices=s)
    assert_bit_equal(tp, base, f"tp_slices={s} logp")
    assert_bit_equal(tpZ, baseZ, f"tp_slices={s} logZ")


def test_from_partials_is_bit_identical(tiny, dev):
    wl, X, W, ids, _ = tiny
    N = wl.n_leaves
    base, baseZ = run(W, X, ids, N, dev)
    with Engine(W.to(dev), n_leaves=N, max_tokens=wl.T) as eng:
        Xd = X.to(dev)
        for s in (1, 2, 4):
            parts = torch.stack([eng.logits_partial(Xd, r * (N // s), N // s) for r in range(s)])
            lp, lz = eng.logprobs_from_partials(parts, ids.to(dev), return_logZ=True)
            eng.check()
            assert_bit_equal(lp, base, f"from {s} partials")
            assert_bit_equal(lz, baseZ, f"logZ from {s} partials")


def test_phase_hint_changes_no_bits(tiny, dev):
    wl, X, W, ids, _ = tiny
    a, _ = run(W, X, ids, wl.n_leaves, dev, phase=1)
    b, _ = run(W, X, ids, wl.n_leaves, dev, phase=2)
    c, _ = run(W, X, ids, wl.n_leaves, dev, phase=0)
    assert_bit_equal(a, b, "prefill vs decode")
    assert_bit_equal(a, c, "prefill vs auto")


@pytest.mark.parametrize("T,H,V,N", [
    (200, 512, 1000, 8),     # ragged rows (2 tiles), ragged vocab tail (104 columns)
    (129, 256, 4224, 2),     # one row past a tile, V = 33 tiles
    (1, 64, 136, 1),         # single row, single leaf, 2 vocab tiles (8-column tail)
    (300, 1024, 777, 4),     # odd V
])
def test_ragged_shapes_match_oracle(dev, T, H, V, N):
    X = inputs.hidden_states(T, H, seed=T + H)
    W = inputs.lm_head(V, H, seed=V + N, std=0.05)
    ids = inputs.uniform_ids(T, V, seed=T)
    logp, logZ = run(W, X, ids, N, dev)
    lp_ref, lz_ref = oracle.logprobs(X, W, ids.numpy())
    assert np.abs(logp.cpu().double().numpy() - lp_ref).max() <= DERIVED_TOL
    assert np.abs(logZ.cpu().double().numpy() - lz_ref).max() <= DERIVED_TOL


def test_two_token_vocab_closed_form(dev):
    # V = 2: logp_y = -log1p(exp(z_other - z_y)), z from the oracle's exact logits.
    T, H = 40, 128
    X = inputs.hidden_states(T, H, seed=5)
    W = inputs.lm_head(2, H, seed=5, std=0.3)
    ids = inputs.uniform_ids(T, 2, seed=5)
    logp, _ = run(W, X, ids, 2, dev)
    z = oracle.logits(X, W)
    y = ids.numpy()
    want = -np.log1p(np.exp(z[np.arange(T), 1 - y] - z[np.arange(T), y]))
    assert np.abs(logp.cpu().double().numpy() - want).max() <= DERIVED_TOL


def test_uniform_logits_give_minus_log_v(dev):
    T, H, V = 64, 256, 4096
    X = inputs.hidden_states(T, H, seed=9)
    W = inputs.lm_head(1, H, seed=9).repeat(V, 1).contiguous()
    ids = inputs.uniform_ids(T, V, seed=9)
    logp, _ = run(W, X, ids, 4, dev)
    assert np.abs(logp.cpu().double().numpy() + math.log(V)).max() <= 1e-5


def test_probabilities_sum_to_one(dev):
    # Score every vocabulary entry of 3 rows: sum_v exp(logp_v) = 1.
    H, V = 256, 4096
    X3 = inputs.hidden_states(3, H, seed=11)
    W = inputs.lm_head(V, H, seed=11, std=0.1)
    X = X3.repeat_interleave(V, dim=0).contiguous()
    ids = torch.arange(V, dtype=torch.int32).repeat(3)
    logp, _ = run(W, X, ids, 4, dev, max_tokens=4096)
    p = torch.exp(logp.cpu().double()).view(3, V).sum(dim=1)
    assert torch.all((p - 1).abs() <= 1e-5), p


def test_bad_ids_give_nan_and_status(tiny, dev):
    wl, X, W, ids, _ = tiny
    bad = ids.clone()
    bad[3], bad[10] = -1, wl.V
    with Engine(W.to(dev), n_leaves=wl.n_leaves, max_tokens=wl.T) as eng:
        logp = eng.logprobs(X.to(dev), bad.to(dev))
        with pytest.raises(LpError) as ei:
            eng.check()
        assert ei.value.code == 1
        eng.clear_status()
        eng.check()
        good = eng.logprobs(X.to(dev), ids.to(dev))
        eng.check()
    lp = logp.cpu()
    assert math.isnan(lp[3]) and math.isnan(lp[10])
    keep = torch.ones(wl.T, dtype=torch.bool)
    keep[3] = keep[10] = False
    assert_bit_equal(lp[keep], good.cpu()[keep], "rows next to a bad id")


def test_empty_batch_is_a_no_op(tiny, dev):
    wl, X, W, ids, _ = tiny
    with Engine(W.to(dev), n_leaves=wl.n_leaves, max_tokens=wl.T) as eng:
        out = eng.logprobs(X[:0].to(dev), ids[:0].to(dev))
        assert out.numel() == 0 and eng.last_launch_count == 0
        w, d3, nv = eng.importance_weights(torch.empty(0, device=dev), torch.empty(0, device=dev))
        eng.check()
        assert d3.item() == 0.0 and nv.item() == 0


def test_importance_weights_match_oracle(dev):
    lp, lm, mask = inputs.synthetic_is_inputs(50000, seed=21)
    W = inputs.lm_head(128, 64, seed=1)
    with Engine(W.to(dev), n_leaves=1, max_tokens=1) as eng:
        w, d3, nv = eng.importance_weights(lp.to(dev), lm.to(dev), mask.to(dev))
        w2, d3b, nv2 = eng.importance_weights(lp.to(dev), lm.to(dev))
        w0, d30, nv0 = eng.importance_weights(lp.to(dev), lp.to(dev), mask.to(dev))
        eng.check()
    w_ref, _, d3_ref, nv_ref = oracle.importance_weights(lp.numpy(), lm.numpy(), mask.numpy())
    np.testing.assert_allclose(w.cpu().double().numpy(), w_ref, rtol=1e-6)
    assert nv.item() == nv_ref
    assert abs(d3.item() - d3_ref) <= 1e-5 * d3_ref
    _, _, d3b_ref, _ = oracle.importance_weights(lp.numpy(), lm.numpy())
    assert nv2.item() == 50000 and abs(d3b.item() - d3b_ref) <= 1e-5 * d3b_ref
    assert_bit_equal(w2, w, "w does not depend on the mask")
    assert d30.item() == 0.0 and nv0.item() == nv_ref
    assert torch.all(w0.cpu() == 1.0)


def test_importance_weights_golden_values(dev, golden_dir):
    import os

    rows = []
    with open(os.path.join(golden_dir, "importance_weights.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#") and not line.startswith("D3"):
                rows.append([float(x) for x in line.split("|")])
    lp = torch.tensor([r[0] for r in rows], dtype=torch.float32)
    lm = torch.tensor([r[1] for r in rows], dtype=torch.float32)
    mask = torch.tensor([int(r[2]) for r in rows], dtype=torch.uint8)
    W = inputs.lm_head(128, 64, seed=1)
    with Engine(W.to(dev), n_leaves=1, max_tokens=1) as eng:
        w, d3, nv = eng.importance_weights(lp.to(dev), lm.to(dev), mask.to(dev))
        eng.check()
    for i, r in enumerate(rows):
        assert float(w[i]) == pytest.approx(r[3], rel=2e-7)
    assert nv.item() == 4
    assert d3.item() == pytest.approx(0.4129839987770457895, rel=1e-6)
    assert bits(w).numel() == len(rows)
