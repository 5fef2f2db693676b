"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle checks.

This module holds no arithmetic of the logprob method itself: it only draws
random numbers and shapes them like the workloads the pages describe (final
hidden states after RMSNorm, a bf16 lm_head, sampled token ids, packed
sequence lengths, a rollout logprob that lags the learner).  Both the CUDA path
and the oracle read the exact same bf16 bytes produced here.

Recipes (all seeded; ``seed`` fully determines the output on a given torch build):
  * hidden states X[T, H]: N(0, 1), then per-row RMSNorm x / sqrt(mean(x^2) + 1e-6)
    (no gain) in fp32, rounded to bf16.
  * lm_head W[V, H]: N(0, 0.02) rounded to bf16 (nn.Linear layout, K-major rows).
  * lagged weights W': bf16(W + N(0, 1e-4)) -- the "weight copy perturbed" that
    stands in for a rollout engine a few updates behind the learner.
  * sampled ids: Gumbel-max draws from given log-probabilities (temperature 1), or
    uniform ids where drawing from the full softmax is too costly.
  * packed sequence lengths: uniform integers in [lo, hi].
"""
from __future__ import annotations

import dataclasses

import torch

__all__ = [
    "Workload", "WORKLOADS", "generator", "hidden_states", "lm_head", "lagged_lm_head",
    "gumbel_max_ids", "uniform_ids", "packed_lengths", "rollout_logprob_noise",
    "synthetic_is_inputs",
]


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape of one synthetic workload (sizes only; no arithmetic)."""

    name: str
    H: int
    V: int
    n_leaves: int
    T: int = 0                      # fixed token count (0: derived from lengths)
    n_seqs: int = 0                 # packed sequences (lengths uniform in [len_lo, len_hi])
    len_lo: int = 0
    len_hi: int = 0
    batch_sizes: tuple = ()         # decode sweep: rows of one token each
    chunk: int = 0                  # row chunk used by the chunked-vs-one-shot check
    tp_slices: tuple = ()           # emulated tensor-parallel splits of K
    seed: int = 1000


# The five workloads: a tiny parity case, two prefill shapes, a decode sweep and
# the importance-weight epilogue at scale.
WORKLOADS = {
    "tiny": Workload("tiny", H=256, V=4096, n_leaves=4, T=64, seed=1000),
    "qwen_prefill": Workload("qwen_prefill", H=2048, V=151936, n_leaves=8, n_seqs=16,
                             len_lo=256, len_hi=2048, seed=1001),
    "ds_prefill": Workload("ds_prefill", H=7168, V=129280, n_leaves=8, T=16384, chunk=2048,
                           tp_slices=(2, 4, 8), seed=1002),
    "ds_decode": Workload("ds_decode", H=7168, V=129280, n_leaves=8,
                          batch_sizes=(1, 7, 32, 128, 256), seed=1003),
    "is_d3": Workload("is_d3", H=4096, V=151936, n_leaves=8, n_seqs=512, len_lo=128,
                      len_hi=8192, seed=1004),
}


def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def hidden_states(T: int, H: int, seed: int, device="cpu") -> torch.Tensor:
    """Final hidden states: N(0,1) rows after RMSNorm (eps 1e-6, no gain), as bf16 [T, H]."""
    g = generator(seed, device)
    x = torch.randn(T, H, generator=g, device=device, dtype=torch.float32)
    x = x * torch.rsqrt(x.pow(2).mean(dim=1, keepdim=True) + 1e-6)
    return x.to(torch.bfloat16).contiguous()


def lm_head(V: int, H: int, seed: int, device="cpu", std: float = 0.02) -> torch.Tensor:
    """lm_head weight W[V, H] ~ N(0, std) as bf16 (row v is the embedding of token v)."""
    g = generator(seed + 7919, device)
    w = torch.randn(V, H, generator=g, device=device, dtype=torch.float32) * std
    return w.to(torch.bfloat16).contiguous()


def lagged_lm_head(W: torch.Tensor, seed: int, std: float = 1e-4) -> torch.Tensor:
    """bf16(W + N(0, std)): a weight copy a few optimizer updates away from W."""
    g = generator(seed + 104729, W.device)
    noise = torch.randn(W.shape, generator=g, device=W.device, dtype=torch.float32) * std
    return (W.float() + noise).to(torch.bfloat16).contiguous()


def gumbel_max_ids(logprobs, seed: int) -> torch.Tensor:
    """Draw one id per row from the categorical distribution with the given log-probs.

    logprobs: [T, V] (numpy or torch, any float dtype).  Returns int32 [T]."""
    lp = torch.as_tensor(logprobs, dtype=torch.float64)
    g = generator(seed + 15485863, "cpu")
    u = torch.rand(lp.shape, generator=g, dtype=torch.float64).clamp_(1e-300, 1.0)
    return torch.argmax(lp - torch.log(-torch.log(u)), dim=1).to(torch.int32)


def uniform_ids(T: int, V: int, seed: int, device="cpu") -> torch.Tensor:
    g = generator(seed + 32452843, device)
    return torch.randint(0, V, (T,), generator=g, device=device, dtype=torch.int32)


def packed_lengths(n_seqs: int, lo: int, hi: int, seed: int) -> list:
    """Sequence lengths uniform in [lo, hi] (inclusive)."""
    g = generator(seed + 49979687, "cpu")
    return [int(v) for v in torch.randint(lo, hi + 1, (n_seqs,), generator=g)]


def rollout_logprob_noise(logp, seed: int, std: float = 1e-3) -> torch.Tensor:
    """A rollout-side logprob mu = logp + N(0, std), as fp32 (tiny workload recipe)."""
    lp = torch.as_tensor(logp, dtype=torch.float64)
    g = generator(seed + 67867967, "cpu")
    return (lp + torch.randn(lp.shape, generator=g, dtype=torch.float64) * std).to(torch.float32)


def synthetic_is_inputs(T: int, seed: int, lag_std: float = 0.05, p_mask: float = 0.9,
                        device="cpu"):
    """Learner / rollout logprobs and a response mask for importance-weight checks.

    log pi: log of uniform(1e-6, 1) probabilities; log mu = log pi + N(0, lag_std);
    mask: 1 with probability p_mask.  Returns (logpi f32[T], logmu f32[T], mask u8[T])."""
    g = generator(seed + 86028121, device)
    u = torch.rand(T, generator=g, device=device, dtype=torch.float32) * (1 - 1e-6) + 1e-6
    logpi = torch.log(u)
    logmu = logpi + torch.randn(T, generator=g, device=device, dtype=torch.float32) * lag_std
    mask = (torch.rand(T, generator=g, device=device) < p_mask).to(torch.uint8)
    return logpi.contiguous(), logmu.contiguous(), mask.contiguous()


def response_batch(n_groups: int, group_size: int, lo: int, hi: int, seed: int,
                   p_reward: float = 0.5):
    """Packed responses for a group-sampled RL batch: lengths uniform in [lo, hi],
    their int64 offsets [B+1] (response i holds tokens [offs[i], offs[i+1])), and 0/1
    rewards drawn with probability p_reward.  CPU tensors."""
    B = n_groups * group_size
    lengths = packed_lengths(B, lo, hi, seed)
    offs = torch.zeros(B + 1, dtype=torch.int64)
    offs[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0)
    g = generator(seed + 15485863, "cpu")
    rewards = (torch.rand(B, generator=g) < p_reward).to(torch.float32)
    return offs, rewards
