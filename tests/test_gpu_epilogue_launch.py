"""The one-launch RL epilogues through the C ABI: importance weights with D3, the acceptance
statistics and the REINFORCE Zero loss.

Each finishes in the last of its blocks to complete: the blocks count themselves on a counter
in the handle, the last one runs the fixed tree over every block partial and resets the
counter for the next call.  So calls of different sizes in a row, and replays of a captured
CUDA graph, must keep giving the bits of the two-step path (block partials, then the fixed
tree over them) that the data-parallel exchange uses (D3: REINFORCE Zero summary, section 3,
a per-update mean over all tokens; IsoExec summary: collectives only transport partials).
"""
import numpy as np
import pytest
import torch

from bit_consistent_logprob_gb300 import Engine, inputs

from gpu_util import assert_bit_equal, require_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def eng():
    dev = require_cuda()
    W = inputs.lm_head(4096, 256, seed=5, device=dev)
    e = Engine(W, n_leaves=4, max_tokens=64)
    yield e
    e.close()


def responses(T, B, seed, device):
    """B responses packed over T tokens (ragged, every one non-empty), rewards in {0, 1}."""
    rng = np.random.default_rng(seed)
    cuts = np.sort(rng.choice(np.arange(1, T), size=B - 1, replace=False))
    offs = np.concatenate([[0], cuts, [T]]).astype(np.int64)
    rewards = rng.integers(0, 2, size=B).astype(np.float32)
    return torch.as_tensor(offs, device=device), torch.as_tensor(rewards, device=device)


def test_sizes_in_a_row_match_the_two_step_path(eng):
    # 1 and 1024 tokens are one block; 1025 a full block and a one-token block; 257 blocks
    # put one value past a warp's 256; 2048 blocks fill one chunk of the final tree exactly,
    # 2049 and 2051 blocks add a second chunk of one and of three, 4097 blocks make three
    # chunks (an odd carry among the chunk results); the counter must start from zero in each
    # call whatever the previous call's block count was.
    dev = require_cuda()
    for T in (5000, 2_100_000, 1, 1024, 1025, 77_777, 262_145, 2_097_152, 2_097_153,
              4_194_305):
        lp, lm, mask = inputs.synthetic_is_inputs(T, seed=T, device=dev)
        w, d3, nv = eng.importance_weights(lp, lm, mask)
        w_p, s, c = eng.importance_weights_partials(lp, lm, mask)
        d3_p, nv_p = eng.d3_from_partials(s, c)
        st = eng.acceptance_stats(lp, lm, mask)
        sums, bmax, cnt = eng.acceptance_stats_partials(lp, lm, mask)
        st_p = eng.acceptance_stats_from_partials(sums, bmax, cnt)
        torch.cuda.synchronize()
        eng.check()
        assert_bit_equal(w, w_p, f"w, T={T}")
        assert_bit_equal(d3, d3_p, f"D3, T={T}")
        assert nv.item() == nv_p.item() == int(mask.sum().item())
        assert_bit_equal(st, st_p, f"acceptance statistics, T={T}")


def test_graph_replays_match_eager(eng):
    dev = require_cuda()
    T, B = 300_001, 96
    lp, lm, mask = inputs.synthetic_is_inputs(T, seed=11, device=dev)
    offs, rewards = responses(T, B, seed=11, device=dev)
    w_e, d3_e, nv_e = eng.importance_weights(lp, lm, mask)
    st_e = eng.acceptance_stats(lp, lm, mask)
    loss_e, wh_e, g_e, adv_e, kept_e = eng.reinforce_zero(lp, lm, offs, rewards, 8, mask=mask,
                                                          tis_cap=2.0)
    torch.cuda.synchronize()
    eng.check()

    w = torch.empty(T, dtype=torch.float32, device=dev)
    d3 = torch.empty(1, dtype=torch.float64, device=dev)
    nv = torch.empty(1, dtype=torch.int64, device=dev)
    st = torch.empty(5, dtype=torch.float64, device=dev)
    wh = torch.empty(T, dtype=torch.float32, device=dev)
    g = torch.empty(T, dtype=torch.float32, device=dev)
    adv = torch.empty(B, dtype=torch.float64, device=dev)

    def step():
        eng.importance_weights(lp, lm, mask, out_w=w, out_d3=d3, out_nvalid=nv)
        eng.acceptance_stats(lp, lm, mask, out=st)
        return eng.reinforce_zero(lp, lm, offs, rewards, 8, mask=mask, tis_cap=2.0,
                                  out_w_hat=wh, out_grad=g, out_adv=adv)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        loss, _, _, _, kept = step()
    for k in range(3):
        for t in (w, d3, nv, st, wh, g, adv, loss, kept):
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        eng.check()
        assert_bit_equal(w, w_e, f"w, replay {k}")
        assert_bit_equal(d3, d3_e, f"D3, replay {k}")
        assert nv.item() == nv_e.item()
        assert_bit_equal(st, st_e, f"statistics, replay {k}")
        assert_bit_equal(loss, loss_e, f"loss, replay {k}")
        assert kept.item() == kept_e.item()
        assert_bit_equal(wh, wh_e, f"w_hat, replay {k}")
        assert_bit_equal(g, g_e, f"gradient, replay {k}")
        assert_bit_equal(adv, adv_e, f"advantages, replay {k}")
