"""Helpers shared by the GPU tests (no arithmetic of the method lives here)."""
import numpy as np
import pytest
import torch

# |logp_gpu - logp_oracle| bound the engine must meet on every workload (nats).
LOGP_TOL = 2e-3


def require_cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device in this environment")
    from bit_consistent_logprob_gb300 import _native

    _native.load(build_if_missing=True)
    return torch.device("cuda:0")


def bits(t: torch.Tensor) -> torch.Tensor:
    """fp32 tensor -> its int32 bit patterns on the CPU (for exact comparisons)."""
    return t.detach().contiguous().cpu().view(torch.int32)


def assert_bit_equal(a: torch.Tensor, b: torch.Tensor, what: str = ""):
    ba, bb = bits(a), bits(b)
    if not torch.equal(ba, bb):
        diff = (ba != bb).nonzero().flatten()
        i = int(diff[0])
        raise AssertionError(
            f"{what}: {diff.numel()} of {ba.numel()} values differ in their bits; first at {i}: "
            f"{a.flatten()[i].item()!r} vs {b.flatten()[i].item()!r}")


def diff_stats(a: torch.Tensor, b: torch.Tensor):
    """max, mean, std of |a - b| and the k3 KL estimator mean(r - 1 - log r), r = exp(a - b)."""
    d = (a.double() - b.double()).cpu()
    r = torch.exp(d)
    k3 = (r - 1 - d).mean().item() if d.numel() else 0.0
    ad = d.abs()
    return dict(max=ad.max().item() if d.numel() else 0.0, mean=ad.mean().item() if d.numel() else 0.0,
                std=ad.std().item() if d.numel() > 1 else 0.0, k3=k3)


def oracle_rows(X, W, ids, rows):
    import oracle

    logp, logZ = oracle.logprobs(X, W, ids.cpu().numpy() if torch.is_tensor(ids) else ids,
                                 rows=np.asarray(rows))
    return logp, logZ
