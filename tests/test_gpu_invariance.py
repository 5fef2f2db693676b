"""Bit-exact invariance of every output row (diff = 0), GPU against GPU.

The acceptance rule is exact equality: the max, mean and std of |delta| and the k3
KL over valid tokens must all be 0 (vLLM blog "Finish RL training faster", section
2).  Each test compares fp32 bit patterns.  The axes follow the same section:
batch independence (size, composition, row position, chunking, packing), phase
consistency (prefill versus one-token decode), parallel layout (emulated TP split
of K), and determinism (run to run, re-initialisation, CUDA graph versus eager,
a concurrent stream occupying SMs, in-place weight updates).
"""
import numpy as np
import pytest
import torch

from bit_consistent_logprob_gb300 import (LP_PHASE_DECODE, LP_PHASE_PREFILL, Engine, inputs)

from gpu_util import assert_bit_equal, diff_stats, require_cuda

pytestmark = pytest.mark.gpu

H, V, N = 1024, 32001, 8          # ragged vocabulary: 251 tiles, the last one 1 column wide
POOL = 4200                       # rows available to build batches from
T_SWEEP = [1, 7, 8, 15, 16, 17, 31, 32, 33, 127, 128, 129, 200, 255, 256, 257, 4096, 4097]


@pytest.fixture(scope="module")
def dev():
    return require_cuda()


@pytest.fixture(scope="module")
def data(dev):
    X = inputs.hidden_states(POOL, H, seed=77, device=dev)
    W = inputs.lm_head(V, H, seed=77, device=dev)
    ids = inputs.uniform_ids(POOL, V, seed=77, device=dev)
    return X, W, ids


@pytest.fixture(scope="module")
def eng(data):
    _, W, _ = data
    e = Engine(W, n_leaves=N, max_tokens=POOL)
    yield e
    e.close()


@pytest.fixture(scope="module")
def solo(eng, data):
    """Every pool row computed alone (T = 1)."""
    X, _, ids = data
    rows = list(range(0, POOL, 97)) + [POOL - 1]
    out = {}
    for r in rows:
        lp, lz = eng.logprobs(X[r:r + 1], ids[r:r + 1], return_logZ=True)
        out[r] = (lp.clone(), lz.clone())
    eng.check()
    return out


def test_row_alone_vs_in_batch_at_any_position(eng, data, solo):
    X, _, ids = data
    rng = np.random.default_rng(1)
    for target in list(solo)[:12]:
        for size in (2, 33, 300, 1500):
            neighbours = rng.choice(POOL, size=size - 1, replace=True)
            for pos in (0, (size - 1) // 2, size - 1):
                order = np.insert(neighbours, pos, target)
                idx = torch.as_tensor(order, device=X.device)
                lp, lz = eng.logprobs(X[idx].contiguous(), ids[idx].contiguous(), return_logZ=True)
                assert_bit_equal(lp[pos:pos + 1], solo[target][0], f"row {target} at {pos}/{size}")
                assert_bit_equal(lz[pos:pos + 1], solo[target][1], f"logZ {target} at {pos}/{size}")
    eng.check()


def test_token_count_sweep(eng, data, solo):
    # Shape thresholds where libraries switch kernels (M < 32 branches, 4096 vs 4097 rows):
    # one path here, so the same row keeps its bits at every batch size.
    X, _, ids = data
    rng = np.random.default_rng(2)
    target = list(solo)[5]
    for T in T_SWEEP:
        pos = int(rng.integers(T))
        order = rng.choice(POOL, size=T, replace=True)
        order[pos] = target
        idx = torch.as_tensor(order, device=X.device)
        lp = eng.logprobs(X[idx].contiguous(), ids[idx].contiguous())
        assert_bit_equal(lp[pos:pos + 1], solo[target][0], f"T={T}")
    eng.check()


def test_combine_layouts_change_no_bits(data, eng, solo):
    # The vocabulary combine picks rows per block (1 to 16) and the per-thread segment
    # length from T; the pairwise tree it evaluates, and so every bit, stay the same.
    X, W, ids = data
    rng = np.random.default_rng(4)
    targets = list(solo)[:4]
    with Engine(W, n_leaves=N, max_tokens=10000) as e:
        for T in (1, 2, 300, 600, 1300, 2500, 5000, 10000):
            order = rng.choice(POOL, size=T, replace=True)
            pos = rng.choice(T, size=min(T, len(targets)), replace=False)
            order[pos] = targets[: len(pos)]
            idx = torch.as_tensor(order, device=X.device)
            lp, lz = e.logprobs(X[idx].contiguous(), ids[idx].contiguous(), return_logZ=True)
            for p_, t in zip(pos, targets):
                assert_bit_equal(lp[p_:p_ + 1], solo[t][0], f"row {t} at T={T}")
                assert_bit_equal(lz[p_:p_ + 1], solo[t][1], f"logZ {t} at T={T}")
        e.check()


def test_chunking_changes_no_bits(data, dev):
    X, W, ids = data
    T = 4097
    ref = None
    for max_tokens in (4097, 1, 7, 128, 1000, 2048):
        if max_tokens == 1:
            Xs, idss = X[:300], ids[:300]  # keep the 1-row chunk run short
        else:
            Xs, idss = X[:T], ids[:T]
        with Engine(W, n_leaves=N, max_tokens=max_tokens) as e:
            lp = e.logprobs(Xs, idss)
            e.check()
        if ref is None:
            ref = lp
        assert_bit_equal(lp, ref[: lp.shape[0]], f"max_tokens={max_tokens}")


@pytest.mark.parametrize("B", [1, 7, 32, 128, 256])
def test_decode_matches_prefill(eng, data, B):
    X, _, ids = data
    prefill = eng.logprobs(X[:2048], ids[:2048], phase=LP_PHASE_PREFILL)
    for start in (0, 1000, 2048 - B):
        dec = eng.logprobs(X[start:start + B], ids[start:start + B], phase=LP_PHASE_DECODE)
        assert_bit_equal(dec, prefill[start:start + B], f"decode B={B} at {start}")
    eng.check()


def test_packed_sequences_vs_each_alone(eng, data):
    X, _, ids = data
    lengths = inputs.packed_lengths(6, 20, 600, seed=3)
    total = sum(lengths)
    packed = eng.logprobs(X[:total], ids[:total])
    off = 0
    for L in lengths:
        alone = eng.logprobs(X[off:off + L], ids[off:off + L])
        assert_bit_equal(alone, packed[off:off + L], f"sequence of {L} tokens at {off}")
        off += L
    eng.check()


@pytest.mark.parametrize("s,T", [(2, 1500), (4, 1500), (8, 1500), (2, 200), (8, 256)])
def test_tp_emulated_split(data, eng, s, T):
    # 1500 rows: a 1024-row and a 476-row pass; 200 and 256 rows: two row tiles, W-sharing pairs
    X, W, ids = data
    base, baseZ = eng.logprobs(X[:T], ids[:T], return_logZ=True)
    with Engine(W, n_leaves=N, tp_slices=s, max_tokens=T) as e:
        lp, lz = e.logprobs(X[:T], ids[:T], return_logZ=True)
        e.check()
    assert_bit_equal(lp, base, f"tp_slices={s}")
    assert_bit_equal(lz, baseZ, f"tp_slices={s} logZ")
    st = diff_stats(lp, base)
    assert st == dict(max=0.0, mean=0.0, std=0.0, k3=0.0)


def test_run_to_run_and_reinit(data, eng):
    X, W, ids = data
    a = eng.logprobs(X[:3000], ids[:3000])
    for _ in range(3):
        assert_bit_equal(eng.logprobs(X[:3000], ids[:3000]), a, "run to run")
    with Engine(W, n_leaves=N, max_tokens=512) as e2:
        assert_bit_equal(e2.logprobs(X[:3000], ids[:3000]), a, "after re-init")
        e2.check()


@pytest.mark.parametrize("T", [1000, 200, 7])  # CTA pairs (8 and 2 row tiles), one CTA per tile
def test_cuda_graph_matches_eager(data, dev, T):
    # The pair launches take their tiles from a counter that a memset node in the graph zeroes
    # before each launch: replaying twice checks that the second replay starts from zero too.
    X, W, ids = data
    with Engine(W, n_leaves=N, max_tokens=T) as e:
        eager = e.logprobs(X[:T], ids[:T])
        out = torch.empty(T, dtype=torch.float32, device=dev)
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            e.logprobs(X[:T], ids[:T], out=out)  # warm-up outside capture
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            e.logprobs(X[:T], ids[:T], out=out)
        for k in range(2):
            out.zero_()
            g.replay()
            torch.cuda.synchronize()
            e.check()
            assert_bit_equal(out, eager, f"graph replay {k} vs eager")


@pytest.mark.parametrize("T", [2000, 256])
def test_concurrent_stream_occupying_sms(data, dev, eng, T):
    X, _, ids = data
    ref = eng.logprobs(X[:T], ids[:T])
    side = torch.cuda.Stream()
    a = torch.randn(8192, 8192, device=dev, dtype=torch.bfloat16)
    with torch.cuda.stream(side):
        for _ in range(6):
            a = (a @ a).clamp_(-1, 1)
    got = eng.logprobs(X[:T], ids[:T])
    torch.cuda.synchronize()
    eng.check()
    assert_bit_equal(got, ref, "with a concurrent stream")


def test_inplace_weight_update(data, dev):
    X, W, ids = data
    T = 800
    W_live = W.clone()
    W_new = inputs.lagged_lm_head(W, seed=5, std=1e-3)
    with Engine(W_live, n_leaves=N, max_tokens=T) as e, Engine(W_new, n_leaves=N, max_tokens=T) as fresh:
        before = e.logprobs(X[:T], ids[:T]).clone()
        W_live.copy_(W_new)  # the weight sync: copy into the original storage
        after = e.logprobs(X[:T], ids[:T])
        want = fresh.logprobs(X[:T], ids[:T])
        e.check()
        fresh.check()
    assert_bit_equal(after, want, "in-place update vs fresh engine")
    assert not torch.equal(before, after)


def test_strided_rows_match_contiguous(data, eng, dev):
    X, _, ids = data
    T = 700
    wide = torch.zeros(T, H + 64, dtype=torch.bfloat16, device=dev)
    wide[:, 32:32 + H] = X[:T]
    view = wide[:, 32:32 + H]  # row stride H + 64, 64-byte offset
    assert view.stride(0) == H + 64
    assert_bit_equal(eng.logprobs(view, ids[:T]), eng.logprobs(X[:T], ids[:T]), "strided X")
    eng.check()


def test_host_buffers_match_device(data, eng):
    X, _, ids = data
    T = 1200
    dev_out = eng.logprobs(X[:T], ids[:T])
    host_out = eng.logprobs_host(X[:T].cpu().pin_memory(), ids[:T].cpu().pin_memory())
    assert_bit_equal(host_out, dev_out, "host API vs device API")


def test_importance_weights_invariance(eng, dev):
    lp, lm, mask = inputs.synthetic_is_inputs(3_000_000, seed=9, device=dev)
    w, d3, nv = eng.importance_weights(lp, lm, mask)
    # per-token weights do not depend on the batch around them
    w_part, _, _ = eng.importance_weights(lp[12345:99999], lm[12345:99999], mask[12345:99999])
    assert_bit_equal(w_part, w[12345:99999], "w of a sub-batch")
    # the host path stages 2^20-token passes: same block tree, same D3 bits
    wh, d3h, nvh = eng.importance_weights_host(lp.cpu(), lm.cpu(), mask.cpu())
    assert_bit_equal(wh, w, "host w")
    assert d3h == d3.item() and nvh == nv.item()
    for _ in range(2):
        _, d3b, _ = eng.importance_weights(lp, lm, mask)
        assert d3b.item() == d3.item()
    eng.check()


@pytest.mark.parametrize("env", ["LP_FORCE_SINGLE_CTA", "LP_FORCE_SHORT_STAGES"])
def test_launch_layout_changes_no_bits(data, eng, env, monkeypatch):
    # CTA pairs (one cta_group::2 MMA over two row tiles) versus one CTA per tile, and 128-K
    # versus 64-K pipeline stages, change only how data moves and who computes a tile.
    X, W, ids = data
    T = 3000
    base, baseZ = eng.logprobs(X[:T], ids[:T], return_logZ=True)
    ent = eng.logprobs_entropy(X[:T], ids[:T])
    monkeypatch.setenv(env, "1")
    with Engine(W, n_leaves=N, max_tokens=T) as e2:
        other, otherZ = e2.logprobs(X[:T], ids[:T], return_logZ=True)
        ent2 = e2.logprobs_entropy(X[:T], ids[:T])
        e2.check()
    assert_bit_equal(other, base, env)
    assert_bit_equal(otherZ, baseZ, env)
    for a, b in zip(ent2, ent):
        assert_bit_equal(a, b, env + " entropy step")


@pytest.mark.parametrize("band", ["1", "3", "7"])
def test_row_bands_change_no_bits(data, eng, band, monkeypatch):
    # Row bands (X rows kept in L2 while the vocabulary sweeps past them) instead of
    # vocabulary bands: only the order in which tiles are handed out changes.
    X, W, ids = data
    T = 3000
    base, baseZ = eng.logprobs(X[:T], ids[:T], return_logZ=True)
    monkeypatch.setenv("LP_BAND_AXIS", "rows")
    monkeypatch.setenv("LP_BAND_ROWS", band)
    with Engine(W, n_leaves=N, max_tokens=T) as e2:
        other, otherZ = e2.logprobs(X[:T], ids[:T], return_logZ=True)
        e2.check()
    assert_bit_equal(other, base, f"row bands of {band}")
    assert_bit_equal(otherZ, baseZ, f"row bands of {band} logZ")


@pytest.mark.parametrize("T", [129, 200, 256, 383])
def test_pairs_with_a_ragged_partner_change_no_bits(data, eng, T, monkeypatch):
    # Calls of 129-256 rows (decode batches of two row tiles) and an odd number of row tiles
    # (383 rows: the last pair's second CTA has no rows) run in CTA pairs; one CTA per tile
    # gives the same bits.
    X, W, ids = data
    base, baseZ = eng.logprobs(X[:T], ids[:T], return_logZ=True)
    monkeypatch.setenv("LP_FORCE_SINGLE_CTA", "1")
    with Engine(W, n_leaves=N, max_tokens=T) as e2:
        other, otherZ = e2.logprobs(X[:T], ids[:T], return_logZ=True)
        e2.check()
    assert_bit_equal(other, base, "LP_FORCE_SINGLE_CTA logp")
    assert_bit_equal(otherZ, baseZ, "LP_FORCE_SINGLE_CTA logZ")
