"""Bit-consistent sampled-token logprob engine for GB300 (sm_103a).

Final hidden states -> lm_head with K cut into N contiguous fp32 leaves combined by a
fixed pairwise tree -> fixed-order log-sum-exp over the vocabulary -> logprob of the
sampled token (optionally the row entropy); the unclipped importance weight
w = exp(log pi - log mu) and D3; acceptance statistics between two logprob vectors; the
REINFORCE Zero loss and its gradient; and the logprob backward (dX, dW).
Every output row is bit-identical across batch size and composition, row position,
prefill versus decode, and an emulated tensor-parallel split of K.

The computation lives in ``liblp.so`` (C ABI: ``include/lp.h``); this package is the
Python binding.  Importing it does not load the library; constructing an ``Engine``
does, and fails loudly if the library is missing.
"""
from ._native import LpError, load as load_library, library_path  # noqa: F401

__all__ = ["Engine", "LpError", "load_library", "library_path", "LP_PHASE_AUTO",
           "LP_PHASE_PREFILL", "LP_PHASE_DECODE", "logprobs_with_grad",
           "visible_with_graph_gradient", "importance_weights_data_parallel",
           "gather_block_partials", "IS_BLOCK", "acceptance_stats_data_parallel",
           "logprobs_vocab_parallel", "gather_vocab_partials"]


def __getattr__(name):
    # Engine imports torch; resolve it lazily so the input generators and the build
    # helper stay importable without touching the GPU stack.
    if name in ("Engine", "LP_PHASE_AUTO", "LP_PHASE_PREFILL", "LP_PHASE_DECODE",
                "logprobs_with_grad", "visible_with_graph_gradient",
                "importance_weights_data_parallel", "gather_block_partials", "IS_BLOCK",
                "acceptance_stats_data_parallel", "logprobs_vocab_parallel",
                "gather_vocab_partials"):
        from . import engine

        return getattr(engine, name)
    raise AttributeError(name)
