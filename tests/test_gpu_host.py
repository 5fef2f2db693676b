"""The host-buffer call against the device call: the same bits for every piece layout.

lp_logprobs_host cuts a batch into row pieces (512 rows, then 8 times the last, up to half the
workspace) that alternate between two halves of the staging workspace, copying the next piece
on a second stream while the current one computes.
Rows are independent of the batch around them (vLLM blog "Finish RL training faster",
section 2: batch independence), so every split must reproduce the device call bit for bit:
one piece, several pieces, more pieces than halves (each half reused), pieces capped by a small
workspace, the serial layout of a workspace under 256 rows, a small call as one piece, strided
host rows, the emulated TP path and the block-FP8 path.
"""
import pytest
import torch

from bit_consistent_logprob_gb300 import Engine, inputs

from gpu_util import assert_bit_equal, require_cuda

pytestmark = pytest.mark.gpu

H, V, N = 512, 8191, 4


@pytest.fixture(scope="module")
def data():
    dev = require_cuda()
    X = inputs.hidden_states(6000, H, seed=21, device=dev)
    W = inputs.lm_head(V, H, seed=21, device=dev)
    ids = inputs.uniform_ids(6000, V, seed=21, device=dev)
    return X, W, ids


def _host(t):
    return t.cpu().pin_memory()


def _compare(eng, X, ids, what):
    lp, lz = eng.logprobs(X, ids, return_logZ=True)
    Xh, idsh = _host(X), _host(ids)
    lzh = torch.empty(X.shape[0], dtype=torch.float32).pin_memory()
    for k in range(2):  # a second call reuses the handle's events and halves
        lph = eng.logprobs_host(Xh, idsh, out_logZ=lzh)
        assert_bit_equal(lph, lp, f"{what}: logp, call {k}")
        assert_bit_equal(lzh, lz, f"{what}: logZ, call {k}")
    eng.check()


@pytest.mark.parametrize("max_tokens,T", [
    (6000, 1),        # one row, one piece
    (6000, 1000),     # the 512-row first piece, then a ragged second in the other half
    (6000, 6000),     # 512, 2944 (a full half), 2544: half 0 reused
    (2600, 5000),     # five pieces, both halves reused, several passes through the workspace
    (1000, 2999),     # pieces capped at a 384-row half: eight pieces
    (200, 777),       # workspace under 256 rows: whole-buffer pieces one after the other
    (256, 256),       # a decode batch filling its workspace: one piece, not two halves
    (1000, 512),      # the largest call that runs as one piece
    (600, 513),       # one row more: 256-row pieces in the two halves
])
def test_host_pieces_match_device(data, max_tokens, T):
    X, W, ids = data
    with Engine(W, n_leaves=N, max_tokens=max_tokens) as eng:
        _compare(eng, X[:T], ids[:T], f"max_tokens={max_tokens} T={T}")


@pytest.mark.parametrize("max_tokens,T", [(256, 256), (1000, 300), (6000, 7)])
def test_host_small_call_is_one_launch(data, max_tokens, T):
    # A call of at most 512 rows that fits the workspace streams W once, like the device call.
    X, W, ids = data
    with Engine(W, n_leaves=N, max_tokens=max_tokens) as eng:
        eng.logprobs(X[:T], ids[:T])
        dev_launches = eng.last_launch_count
        eng.logprobs_host(_host(X[:T]), _host(ids[:T]))
        assert eng.last_launch_count == dev_launches
        eng.check()


def test_host_strided_rows(data):
    X, W, ids = data
    T = 2500
    wide = torch.zeros(T, H + 64, dtype=torch.bfloat16)
    wide[:, 32:32 + H] = X[:T].cpu()
    view = wide.pin_memory()[:, 32:32 + H]
    with Engine(W, n_leaves=N, max_tokens=4096) as eng:
        lp = eng.logprobs(X[:T], ids[:T])
        got = eng.logprobs_host(view, _host(ids[:T]))
        eng.check()
    assert_bit_equal(got, lp, "strided host rows")


def test_host_tp_slices(data):
    X, W, ids = data
    with Engine(W, n_leaves=N, tp_slices=2, max_tokens=5000) as eng:
        _compare(eng, X[:5000], ids[:5000], "tp_slices=2 (pieces capped at 1024-row passes)")


def test_host_fp8(data):
    X, W, ids = data
    with Engine(W, n_leaves=N, max_tokens=3000, fp8=True) as eng:
        _compare(eng, X[:3000], ids[:3000], "block FP8")
