"""PyTorch-facing wrapper of the C ABI: device memory and streams come from torch,
every computation runs in the library's CUDA kernels."""
from __future__ import annotations

import ctypes

import torch

from . import _native
from ._native import LP_PHASE_AUTO, LP_PHASE_DECODE, LP_PHASE_PREFILL, LpConfig, LpError

IS_BLOCK = 1024  # tokens per D3 block (LP_IS_BLOCK in include/lp.h)

__all__ = ["Engine", "LpError", "LP_PHASE_AUTO", "LP_PHASE_PREFILL", "LP_PHASE_DECODE"]


def _stream_ptr(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


class _DeviceArray:
    """A borrowed device buffer described by the CUDA array interface (no copy)."""

    def __init__(self, ptr, shape, typestr):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (int(ptr), False), "version": 3, "strides": None}


def _device_view(ptr, shape, typestr, device):
    with torch.cuda.device(device):
        return torch.as_tensor(_DeviceArray(ptr, shape, typestr), device=device)


def _require(t: torch.Tensor, name: str, dtype, ndim: int, device_type="cuda"):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must be {ndim}-D, got shape {tuple(t.shape)}")
    if t.device.type != device_type:
        raise ValueError(f"{name} must live on {device_type}, got {t.device}")


class Engine:
    """Bit-consistent sampled-token logprob engine for one lm_head.

    W: bf16 [V, H] CUDA tensor (referenced, not copied: in-place updates are seen).
    n_leaves: N contiguous K leaves combined by the fixed pairwise tree (1, 2, 4, 8).
    tp_slices: emulated tensor-parallel split of K for ``logprobs`` (1 = fused path).
    max_tokens: rows per pass; sizes the workspace.
    fp8: block-FP8 (W8A8) handle: W is quantised to e4m3 in 128 x 128 blocks at construction
    (and by ``fp8_requantize``), each batch of X in 1 x 128 blocks per call.
    """

    def __init__(self, W: torch.Tensor, n_leaves: int = 8, tp_slices: int = 1,
                 max_tokens: int = 16384, stream=None, fp8: bool = False):
        _require(W, "W", torch.bfloat16, 2)
        if not W.is_contiguous():
            raise ValueError("W must be contiguous")
        self._lib = _native.load()
        self.V, self.H = int(W.shape[0]), int(W.shape[1])
        self.n_leaves, self.tp_slices, self.max_tokens = int(n_leaves), int(tp_slices), int(max_tokens)
        self._W = W
        cfg = LpConfig(self.H, self.V, self.n_leaves, self.tp_slices, self.max_tokens)
        h = ctypes.c_void_p()
        with torch.cuda.device(W.device):
            init = self._lib.lp_init_fp8 if fp8 else self._lib.lp_init
            _native.check(init(ctypes.byref(cfg), _ptr(W), _stream_ptr(stream), ctypes.byref(h)))
        self._h = h
        self.device = W.device
        self.fp8 = bool(fp8)

    # ------------------------------------------------------------------ logprobs
    def logprobs(self, X: torch.Tensor, ids: torch.Tensor, out: torch.Tensor = None,
                 out_logZ: torch.Tensor = None, return_logZ: bool = False,
                 phase: int = LP_PHASE_AUTO, stream=None):
        """logp[t] = z[t, ids[t]] - logZ[t] for X bf16 [T, H] (row stride may exceed H)."""
        _require(X, "X", torch.bfloat16, 2)
        _require(ids, "ids", torch.int32, 1)
        T = int(X.shape[0])
        if X.shape[1] != self.H or X.stride(1) != 1:
            raise ValueError("X must be [T, H] with unit column stride")
        if ids.shape[0] != T or not ids.is_contiguous():
            raise ValueError("ids must be a contiguous [T] tensor")
        if out is None:
            out = torch.empty(T, dtype=torch.float32, device=X.device)
        if return_logZ and out_logZ is None:
            out_logZ = torch.empty(T, dtype=torch.float32, device=X.device)
        ldx = X.stride(0) if T > 1 else self.H
        _native.check(self._lib.lp_logprobs(self._h, _ptr(X), ldx, _ptr(ids), T, _ptr(out),
                                            _ptr(out_logZ), int(phase), _stream_ptr(stream)))
        return (out, out_logZ) if (return_logZ or out_logZ is not None) else out

    def logprobs_entropy(self, X: torch.Tensor, ids: torch.Tensor, out: torch.Tensor = None,
                         out_logZ: torch.Tensor = None, out_entropy: torch.Tensor = None,
                         phase: int = LP_PHASE_AUTO, stream=None):
        """(logp, logZ, entropy) fp32 [T]: logprobs plus each row's softmax entropy."""
        _require(X, "X", torch.bfloat16, 2)
        _require(ids, "ids", torch.int32, 1)
        T = int(X.shape[0])
        if X.shape[1] != self.H or X.stride(1) != 1:
            raise ValueError("X must be [T, H] with unit column stride")
        if ids.shape[0] != T or not ids.is_contiguous():
            raise ValueError("ids must be a contiguous [T] tensor")
        dev = X.device
        out = torch.empty(T, dtype=torch.float32, device=dev) if out is None else out
        out_logZ = torch.empty(T, dtype=torch.float32, device=dev) if out_logZ is None else out_logZ
        if out_entropy is None:
            out_entropy = torch.empty(T, dtype=torch.float32, device=dev)
        ldx = X.stride(0) if T > 1 else self.H
        _native.check(self._lib.lp_logprobs_entropy(
            self._h, _ptr(X), ldx, _ptr(ids), T, _ptr(out), _ptr(out_logZ), _ptr(out_entropy),
            int(phase), _stream_ptr(stream)))
        return out, out_logZ, out_entropy

    # ------------------------------------------------------------------ block FP8
    def fp8_requantize(self, stream=None) -> None:
        """Re-quantise the referenced bf16 lm_head (after an in-place update)."""
        _native.check(self._lib.lp_fp8_requantize(self._h, _stream_ptr(stream)))

    def fp8_weights(self):
        """(wq uint8 [V, H], sw fp32 [ceil(V/128), H/128]): copies of the handle's e4m3 lm_head."""
        wq, sw = ctypes.c_void_p(), ctypes.c_void_p()
        _native.check(self._lib.lp_fp8_weights(self._h, ctypes.byref(wq), ctypes.byref(sw)))
        nvb, nkb = (self.V + 127) // 128, self.H // 128
        return (_device_view(wq.value, (self.V, self.H), "|u1", self.device).clone(),
                _device_view(sw.value, (nvb, nkb), "<f4", self.device).clone())

    def fp8_quantize_x(self, X: torch.Tensor, stream=None):
        """The activation rule alone: (xq uint8 [T, H], sx fp32 [T, H/128])."""
        _require(X, "X", torch.bfloat16, 2)
        T = int(X.shape[0])
        xq = torch.empty(T, self.H, dtype=torch.uint8, device=X.device)
        sx = torch.empty(T, self.H // 128, dtype=torch.float32, device=X.device)
        ldx = X.stride(0) if T > 1 else self.H
        _native.check(self._lib.lp_fp8_quantize_x(self._h, _ptr(X), ldx, T, _ptr(xq), _ptr(sx),
                                                  _stream_ptr(stream)))
        return xq, sx

    # ------------------------------------------------------------------ backward
    def backward_reserve(self, max_rows: int) -> None:
        """Allocate the backward's bf16 logit-gradient buffer for chunks of max_rows rows."""
        with torch.cuda.device(self.device):
            _native.check(self._lib.lp_backward_reserve(self._h, int(max_rows)))

    def logprobs_backward(self, X: torch.Tensor, ids: torch.Tensor, logZ: torch.Tensor,
                          grad_logp: torch.Tensor, need_dX: bool = True, need_dW: bool = True,
                          dX: torch.Tensor = None, dW: torch.Tensor = None,
                          accumulate: bool = False, stream=None):
        """(dX fp32 [T, H], dW fp32 [V, H]) for upstream gradient grad_logp = dL/dlogp."""
        _require(X, "X", torch.bfloat16, 2)
        _require(ids, "ids", torch.int32, 1)
        _require(logZ, "logZ", torch.float32, 1)
        _require(grad_logp, "grad_logp", torch.float32, 1)
        T = int(X.shape[0])
        if X.shape[1] != self.H or X.stride(1) != 1:
            raise ValueError("X must be [T, H] with unit column stride")
        for t, name in ((ids, "ids"), (logZ, "logZ"), (grad_logp, "grad_logp")):
            if t.shape[0] != T or not t.is_contiguous():
                raise ValueError(f"{name} must be a contiguous [T] tensor")
        dev = X.device
        if need_dX and dX is None:
            dX = torch.empty(T, self.H, dtype=torch.float32, device=dev)
        if need_dW and dW is None:
            dW = torch.empty(self.V, self.H, dtype=torch.float32, device=dev)
            accumulate = False
        ldx = X.stride(0) if T > 1 else self.H
        _native.check(self._lib.lp_logprobs_backward(
            self._h, _ptr(X), ldx, _ptr(ids), _ptr(logZ), _ptr(grad_logp), T,
            _ptr(dX if need_dX else None), _ptr(dW if need_dW else None), int(bool(accumulate)),
            _stream_ptr(stream)))
        return (dX if need_dX else None), (dW if need_dW else None)

    def logprobs_host(self, X: torch.Tensor, ids: torch.Tensor, out: torch.Tensor = None,
                      out_logZ: torch.Tensor = None, stream=None):
        """Host-memory variant: X, ids, out live in (preferably pinned) CPU memory."""
        _require(X, "X", torch.bfloat16, 2, "cpu")
        _require(ids, "ids", torch.int32, 1, "cpu")
        T = int(X.shape[0])
        if X.shape[1] != self.H or X.stride(1) != 1 or ids.shape[0] != T:
            raise ValueError("X must be [T, H] with unit column stride; ids [T]")
        if out is None:
            out = torch.empty(T, dtype=torch.float32, pin_memory=True)
        ldx = X.stride(0) if T > 1 else self.H
        with torch.cuda.device(self.device):
            _native.check(self._lib.lp_logprobs_host(self._h, _ptr(X), ldx, _ptr(ids), T,
                                                     _ptr(out), _ptr(out_logZ),
                                                     _stream_ptr(stream)))
        return out

    def logits_partial(self, X: torch.Tensor, leaf_begin: int, leaf_count: int,
                       out: torch.Tensor = None, stream=None) -> torch.Tensor:
        """fp32 [T, V] tree node over leaves [leaf_begin, leaf_begin + leaf_count)."""
        _require(X, "X", torch.bfloat16, 2)
        T = int(X.shape[0])
        if out is None:
            ldo = (self.V + 3) // 4 * 4
            out = torch.empty(T, ldo, dtype=torch.float32, device=X.device)[:, : self.V]
        ldx = X.stride(0) if T > 1 else self.H
        ldo = out.stride(0) if T > 1 else (self.V + 3) // 4 * 4
        _native.check(self._lib.lp_logits_partial(self._h, _ptr(X), ldx, T, int(leaf_begin),
                                                  int(leaf_count), _ptr(out), ldo,
                                                  _stream_ptr(stream)))
        return out

    def logprobs_from_partials(self, partials: torch.Tensor, ids: torch.Tensor,
                               out: torch.Tensor = None, out_logZ: torch.Tensor = None,
                               return_logZ: bool = False, stream=None):
        """Finish from gathered tree nodes: partials fp32 [n_parts, T, ldp] (ldp >= V)."""
        _require(partials, "partials", torch.float32, 3)
        _require(ids, "ids", torch.int32, 1)
        n_parts, T = int(partials.shape[0]), int(partials.shape[1])
        if partials.stride(2) != 1:
            raise ValueError("partials must have unit stride in the vocabulary axis")
        if out is None:
            out = torch.empty(T, dtype=torch.float32, device=partials.device)
        if return_logZ and out_logZ is None:
            out_logZ = torch.empty(T, dtype=torch.float32, device=partials.device)
        _native.check(self._lib.lp_logprobs_from_partials(
            self._h, _ptr(partials), n_parts, partials.stride(0), partials.stride(1), _ptr(ids), T,
            _ptr(out), _ptr(out_logZ), _stream_ptr(stream)))
        return (out, out_logZ) if (return_logZ or out_logZ is not None) else out

    # ------------------------------------------------------------------ IS / D3
    def importance_weights(self, logp_pi: torch.Tensor, logp_mu: torch.Tensor,
                           mask: torch.Tensor = None, out_w: torch.Tensor = None,
                           out_d3: torch.Tensor = None, out_nvalid: torch.Tensor = None,
                           stream=None):
        """(w fp32 [T], D3 fp64 [1], n_valid int64 [1]) -- all on the device, no sync."""
        _require(logp_pi, "logp_pi", torch.float32, 1)
        _require(logp_mu, "logp_mu", torch.float32, 1)
        T = int(logp_pi.shape[0])
        if logp_mu.shape[0] != T:
            raise ValueError("logp_pi and logp_mu must have the same length")
        if mask is not None:
            _require(mask, "mask", torch.uint8, 1)
            if mask.shape[0] != T:
                raise ValueError("mask must have length T")
        dev = logp_pi.device
        if out_w is None:
            out_w = torch.empty(T, dtype=torch.float32, device=dev)
        if out_d3 is None:
            out_d3 = torch.empty(1, dtype=torch.float64, device=dev)
        if out_nvalid is None:
            out_nvalid = torch.empty(1, dtype=torch.int64, device=dev)
        _native.check(self._lib.lp_importance_weights(
            self._h, _ptr(logp_pi), _ptr(logp_mu), _ptr(mask), T, _ptr(out_w), _ptr(out_d3),
            _ptr(out_nvalid), _stream_ptr(stream)))
        return out_w, out_d3, out_nvalid

    def vocab_partials(self, X: torch.Tensor, ids_local: torch.Tensor, stream=None):
        """This vocabulary slice's share of a vocabulary-parallel logprob: (ms fp32
        [ceil(V/64), T, 2]: per-tile (max, sum-exp); zy fp32 [T]: sampled logit, defined where
        0 <= ids_local < V).  The handle is opened over the slice; ids_local = id - v0."""
        _require(X, "X", torch.bfloat16, 2)
        _require(ids_local, "ids_local", torch.int32, 1)
        T = int(X.shape[0])
        if X.shape[1] != self.H or X.stride(1) != 1:
            raise ValueError("X must be [T, H] with unit column stride")
        if ids_local.shape[0] != T or not ids_local.is_contiguous():
            raise ValueError("ids_local must be a contiguous [T] tensor")
        nt = (self.V + 63) // 64
        ms = torch.empty(nt, T, 2, dtype=torch.float32, device=X.device)
        zy = torch.empty(T, dtype=torch.float32, device=X.device)
        ldx = X.stride(0) if T > 1 else self.H
        _native.check(self._lib.lp_vocab_partials(self._h, _ptr(X), ldx, _ptr(ids_local), T,
                                                  _ptr(ms), T, _ptr(zy), _stream_ptr(stream)))
        return ms, zy

    def logprobs_from_vocab_partials(self, V_full: int, ms: torch.Tensor, zy: torch.Tensor,
                                     ids: torch.Tensor, return_logZ: bool = False, stream=None):
        """logp (and logZ) over the full vocabulary from gathered tile partials
        ms [ceil(V_full/64), T, 2] (vocabulary order) and owner-picked zy [T]."""
        _require(ms, "ms", torch.float32, 3)
        _require(zy, "zy", torch.float32, 1)
        _require(ids, "ids", torch.int32, 1)
        T = int(zy.shape[0])
        if ms.shape != ((int(V_full) + 63) // 64, T, 2) or not ms.is_contiguous():
            raise ValueError("ms must be a contiguous [ceil(V_full/64), T, 2] tensor")
        out = torch.empty(T, dtype=torch.float32, device=zy.device)
        out_logZ = torch.empty(T, dtype=torch.float32, device=zy.device) if return_logZ else None
        _native.check(self._lib.lp_logprobs_from_vocab_partials(
            self._h, int(V_full), _ptr(ms), T, _ptr(zy), _ptr(ids), T, _ptr(out), _ptr(out_logZ),
            _stream_ptr(stream)))
        return (out, out_logZ) if return_logZ else out

    def importance_weights_partials(self, logp_pi: torch.Tensor, logp_mu: torch.Tensor,
                                    mask: torch.Tensor = None, stream=None):
        """(w fp32 [T], block sums fp64 [nb], block counts int64 [nb]), nb = ceil(T / 1024):
        this rank's share of a data-parallel D3 (see ``d3_from_partials``)."""
        _require(logp_pi, "logp_pi", torch.float32, 1)
        _require(logp_mu, "logp_mu", torch.float32, 1)
        T = int(logp_pi.shape[0])
        if logp_mu.shape[0] != T:
            raise ValueError("logp_pi and logp_mu must have the same length")
        if mask is not None:
            _require(mask, "mask", torch.uint8, 1)
            if mask.shape[0] != T:
                raise ValueError("mask must have length T")
        dev = logp_pi.device
        nb = (T + IS_BLOCK - 1) // IS_BLOCK
        w = torch.empty(T, dtype=torch.float32, device=dev)
        blk_sum = torch.empty(nb, dtype=torch.float64, device=dev)
        blk_cnt = torch.empty(nb, dtype=torch.int64, device=dev)
        _native.check(self._lib.lp_importance_weights_partials(
            self._h, _ptr(logp_pi), _ptr(logp_mu), _ptr(mask), T, _ptr(w), _ptr(blk_sum),
            _ptr(blk_cnt), _stream_ptr(stream)))
        return w, blk_sum, blk_cnt

    def d3_from_partials(self, blk_sum: torch.Tensor, blk_cnt: torch.Tensor, stream=None):
        """(D3 fp64 [1], n_valid int64 [1]) from gathered 1024-token block partials, in
        stream order, by the same fixed tree as ``importance_weights``."""
        _require(blk_sum, "blk_sum", torch.float64, 1)
        _require(blk_cnt, "blk_cnt", torch.int64, 1)
        nb = int(blk_sum.shape[0])
        if blk_cnt.shape[0] != nb or not (blk_sum.is_contiguous() and blk_cnt.is_contiguous()):
            raise ValueError("blk_sum and blk_cnt must be contiguous and of the same length")
        out_d3 = torch.empty(1, dtype=torch.float64, device=blk_sum.device)
        out_nvalid = torch.empty(1, dtype=torch.int64, device=blk_sum.device)
        _native.check(self._lib.lp_d3_from_partials(
            self._h, _ptr(blk_sum), _ptr(blk_cnt), nb, _ptr(out_d3), _ptr(out_nvalid),
            _stream_ptr(stream)))
        return out_d3, out_nvalid

    def acceptance_stats(self, logp_a: torch.Tensor, logp_b: torch.Tensor,
                         mask: torch.Tensor = None, out: torch.Tensor = None, stream=None):
        """fp64 [5] on the device: max, mean and std of |a - b|, k3, n_valid (no sync)."""
        _require(logp_a, "logp_a", torch.float32, 1)
        _require(logp_b, "logp_b", torch.float32, 1)
        T = int(logp_a.shape[0])
        if logp_b.shape[0] != T:
            raise ValueError("logp_a and logp_b must have the same length")
        if mask is not None:
            _require(mask, "mask", torch.uint8, 1)
            if mask.shape[0] != T:
                raise ValueError("mask must have length T")
        if out is None:
            out = torch.empty(_native.LP_STAT_COUNT, dtype=torch.float64, device=logp_a.device)
        _native.check(self._lib.lp_acceptance_stats(
            self._h, _ptr(logp_a), _ptr(logp_b), _ptr(mask), T, _ptr(out), _stream_ptr(stream)))
        return out

    def acceptance_stats_partials(self, logp_a: torch.Tensor, logp_b: torch.Tensor,
                                  mask: torch.Tensor = None, stream=None):
        """This rank's 1024-token block partials of the acceptance statistics:
        (sums fp64 [3, nb]: sum |d|, sum d^2, sum k3 term; max fp32 [nb]; counts int64 [nb])."""
        _require(logp_a, "logp_a", torch.float32, 1)
        _require(logp_b, "logp_b", torch.float32, 1)
        T = int(logp_a.shape[0])
        if logp_b.shape[0] != T:
            raise ValueError("logp_a and logp_b must have the same length")
        if mask is not None:
            _require(mask, "mask", torch.uint8, 1)
            if mask.shape[0] != T:
                raise ValueError("mask must have length T")
        dev = logp_a.device
        nb = (T + IS_BLOCK - 1) // IS_BLOCK
        sums = torch.empty(3, nb, dtype=torch.float64, device=dev)
        bmax = torch.empty(nb, dtype=torch.float32, device=dev)
        cnts = torch.empty(nb, dtype=torch.int64, device=dev)
        _native.check(self._lib.lp_acceptance_stats_partials(
            self._h, _ptr(logp_a), _ptr(logp_b), _ptr(mask), T, _ptr(sums), _ptr(bmax),
            _ptr(cnts), _stream_ptr(stream)))
        return sums, bmax, cnts

    def acceptance_stats_from_partials(self, sums: torch.Tensor, bmax: torch.Tensor,
                                       cnts: torch.Tensor, stream=None):
        """fp64 [5] as ``acceptance_stats``, from gathered block partials in stream order."""
        _require(sums, "sums", torch.float64, 2)
        _require(bmax, "bmax", torch.float32, 1)
        _require(cnts, "cnts", torch.int64, 1)
        nb = int(cnts.shape[0])
        if sums.shape != (3, nb) or bmax.shape[0] != nb or not (
                sums.is_contiguous() and bmax.is_contiguous() and cnts.is_contiguous()):
            raise ValueError("sums [3, nb], bmax [nb] and cnts [nb] must be contiguous")
        out = torch.empty(_native.LP_STAT_COUNT, dtype=torch.float64, device=sums.device)
        _native.check(self._lib.lp_acceptance_stats_from_partials(
            self._h, _ptr(sums), _ptr(bmax), _ptr(cnts), nb, _ptr(out), _stream_ptr(stream)))
        return out

    def reinforce_zero(self, logp_pi: torch.Tensor, logp_mu: torch.Tensor,
                       seq_offsets: torch.Tensor, rewards: torch.Tensor, group_size: int,
                       mask: torch.Tensor = None, tis_cap: float = None,
                       token_gate: tuple = None, seq_gate: tuple = None,
                       out_w_hat: torch.Tensor = None, out_grad: torch.Tensor = None,
                       out_adv: torch.Tensor = None, stream=None):
        """REINFORCE Zero loss over responses packed at ``seq_offsets`` ([B+1] int64).

        tis_cap: TIS cap C (w_hat = min(w, C)); token_gate: (lo, hi) bounds on
        d = log pi - log mu; seq_gate: (lo, hi) bounds on a response's sum of d.
        Returns (loss fp64 [1], w_hat fp32 [T], grad fp32 [T] = dL/dlog pi,
        adv fp64 [B], n_kept int64 [1]), all on the device, no sync."""
        _require(logp_pi, "logp_pi", torch.float32, 1)
        _require(logp_mu, "logp_mu", torch.float32, 1)
        _require(seq_offsets, "seq_offsets", torch.int64, 1)
        _require(rewards, "rewards", torch.float32, 1)
        T = int(logp_pi.shape[0])
        B = int(rewards.shape[0])
        if logp_mu.shape[0] != T or seq_offsets.shape[0] != B + 1:
            raise ValueError("need logp_mu of length T and seq_offsets of length B + 1")
        if mask is not None:
            _require(mask, "mask", torch.uint8, 1)
            if mask.shape[0] != T:
                raise ValueError("mask must have length T")
        opt = _native.LpRzOptions()
        if tis_cap is not None:
            opt.flags |= _native.LP_RZ_TIS
            opt.tis_cap = float(tis_cap)
        if token_gate is not None:
            opt.flags |= _native.LP_RZ_TOKEN_GATE
            opt.token_log_lo, opt.token_log_hi = (float(v) for v in token_gate)
        if seq_gate is not None:
            opt.flags |= _native.LP_RZ_SEQ_GATE
            opt.seq_log_lo, opt.seq_log_hi = (float(v) for v in seq_gate)
        dev = logp_pi.device
        if out_w_hat is None:
            out_w_hat = torch.empty(T, dtype=torch.float32, device=dev)
        if out_grad is None:
            out_grad = torch.empty(T, dtype=torch.float32, device=dev)
        if out_adv is None:
            out_adv = torch.empty(B, dtype=torch.float64, device=dev)
        loss = torch.empty(1, dtype=torch.float64, device=dev)
        n_kept = torch.empty(1, dtype=torch.int64, device=dev)
        _native.check(self._lib.lp_reinforce_zero(
            self._h, _ptr(logp_pi), _ptr(logp_mu), _ptr(mask), T, _ptr(seq_offsets), B,
            _ptr(rewards), int(group_size), ctypes.byref(opt), _ptr(out_w_hat), _ptr(out_grad),
            _ptr(out_adv), _ptr(loss), _ptr(n_kept), _stream_ptr(stream)))
        return loss, out_w_hat, out_grad, out_adv, n_kept

    def importance_weights_host(self, logp_pi: torch.Tensor, logp_mu: torch.Tensor,
                                mask: torch.Tensor = None, out_w: torch.Tensor = None,
                                stream=None):
        """Host-memory variant: returns (w fp32 [T] on the host, D3 float, n_valid int)."""
        _require(logp_pi, "logp_pi", torch.float32, 1, "cpu")
        _require(logp_mu, "logp_mu", torch.float32, 1, "cpu")
        T = int(logp_pi.shape[0])
        if mask is not None:
            _require(mask, "mask", torch.uint8, 1, "cpu")
        if out_w is None:
            out_w = torch.empty(T, dtype=torch.float32, pin_memory=True)
        d3 = ctypes.c_double()
        nv = ctypes.c_int64()
        with torch.cuda.device(self.device):
            _native.check(self._lib.lp_importance_weights_host(
                self._h, _ptr(logp_pi), _ptr(logp_mu), _ptr(mask), T, _ptr(out_w),
                ctypes.byref(d3), ctypes.byref(nv), _stream_ptr(stream)))
        return out_w, d3.value, nv.value

    # ------------------------------------------------------------------ profiling
    def profile_enable(self, enable: bool = True) -> None:
        """Bracket every leaf-GEMM launch with CUDA events on its stream."""
        _native.check(self._lib.lp_profile_enable(self._h, int(bool(enable))))

    def profile_read_kind(self, kind: int):
        """(total milliseconds, count) of one timed kind (_native.LP_PROFILE_*) since the last
        profile_read, without clearing; synchronises."""
        ms = ctypes.c_double()
        n = ctypes.c_int32()
        _native.check(self._lib.lp_profile_read_kind(self._h, int(kind), ctypes.byref(ms),
                                                     ctypes.byref(n)))
        return ms.value, n.value

    def profile_read(self):
        """(total leaf-GEMM milliseconds, launches) since the last read; synchronises."""
        ms = ctypes.c_double()
        n = ctypes.c_int32()
        _native.check(self._lib.lp_profile_read(self._h, ctypes.byref(ms), ctypes.byref(n)))
        return ms.value, n.value

    # ------------------------------------------------------------------ status
    def check(self) -> None:
        """Synchronise and raise LpError if a kernel flagged a bad id or a wait timeout."""
        _native.check(self._lib.lp_check(self._h))

    def selftest_wait_timeout(self, timeout_us: int = 1000, stream=None) -> None:
        """Run the bounded-wait self-test (raises the sticky timeout status; see lp.h)."""
        _native.check(self._lib.lp_selftest_wait_timeout(self._h, int(timeout_us),
                                                         _stream_ptr(stream)))

    def clear_status(self, stream=None) -> None:
        _native.check(self._lib.lp_clear_status(self._h, _stream_ptr(stream)))

    @property
    def workspace_bytes(self) -> int:
        return int(self._lib.lp_workspace_bytes(self._h))

    @property
    def last_launch_count(self) -> int:
        return int(self._lib.lp_last_launch_count(self._h))

    def close(self) -> None:
        if getattr(self, "_h", None):
            self._lib.lp_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


class _Logprobs(torch.autograd.Function):
    """Forward values from the bit-consistent kernel; backward from lp_logprobs_backward."""

    @staticmethod
    def forward(ctx, X, W, ids, engine):
        logp, logZ = engine.logprobs(X, ids, return_logZ=True)
        ctx.engine = engine
        ctx.save_for_backward(X, ids, logZ)
        ctx.mark_non_differentiable(logZ)
        return logp

    @staticmethod
    def backward(ctx, grad):
        X, ids, logZ = ctx.saved_tensors
        need_dX, need_dW = ctx.needs_input_grad[0], ctx.needs_input_grad[1]
        dX, dW = ctx.engine.logprobs_backward(X, ids, logZ, grad.contiguous().float(),
                                              need_dX=need_dX, need_dW=need_dW)
        return (dX.to(X.dtype) if dX is not None else None,
                dW.to(ctx.engine._W.dtype) if dW is not None else None, None, None)


def logprobs_with_grad(engine: "Engine", X: torch.Tensor, W: torch.Tensor,
                       ids: torch.Tensor) -> torch.Tensor:
    """Differentiable sampled-token logprobs: the values are the engine's bit-consistent
    forward; gradients with respect to X and W come from the engine's backward.  W must be
    the tensor the engine was built on (it is referenced, not copied)."""
    if W.data_ptr() != engine._W.data_ptr():
        raise ValueError("W must be the engine's lm_head tensor")
    engine.backward_reserve(min(int(X.shape[0]), engine.max_tokens) or 1)
    return _Logprobs.apply(X, W, ids, engine)


def visible_with_graph_gradient(visible: torch.Tensor, graph: torch.Tensor) -> torch.Tensor:
    """visible + (graph - graph.detach()): the value of ``visible`` (e.g. the bit-consistent
    kernel's logprobs) with the gradient of ``graph`` (any differentiable computation of the
    same quantity), the form the pages give for attaching a training graph's backward to an
    inference kernel's forward values (vLLM blog "Finish RL training faster", section 3.1).
    ``logprobs_with_grad`` does the same job with the engine's own backward."""
    if visible.shape != graph.shape:
        raise ValueError("visible and graph must have the same shape")
    return visible.detach() + (graph - graph.detach())


def gather_block_partials(*arrays: torch.Tensor, group=None):
    """All-gather every rank's per-block partial arrays and concatenate them in rank order.

    Each array has the rank's block count as its last dimension (the leading dimensions must
    agree across ranks).  The collective only moves the values (padded to the longest rank's
    block count, then trimmed); it never adds them, so the gathered blocks are bit-identical
    to the ones one rank would have computed for the whole stream.  Returns one tensor per
    array.
    """
    import torch.distributed as dist

    world = dist.get_world_size(group)
    nb = arrays[0].shape[-1]
    n = torch.tensor([nb], dtype=torch.int64, device=arrays[0].device)
    sizes = [torch.zeros_like(n) for _ in range(world)]
    dist.all_gather(sizes, n, group=group)
    sizes = [int(x.item()) for x in sizes]
    m = max(sizes)
    out = []
    for t in arrays:
        if t.shape[-1] != nb:
            raise ValueError("every partial array must have one entry per block")
        pad = torch.zeros(*t.shape[:-1], m, dtype=t.dtype, device=t.device)
        pad[..., :nb] = t
        parts = [torch.empty_like(pad) for _ in range(world)]
        dist.all_gather(parts, pad.contiguous(), group=group)
        out.append(torch.cat([x[..., :k] for x, k in zip(parts, sizes)], dim=-1).contiguous())
    return tuple(out)


def importance_weights_data_parallel(engine: "Engine", logp_pi: torch.Tensor,
                                     logp_mu: torch.Tensor, mask: torch.Tensor = None,
                                     group=None):
    """(w [T], D3 [1], n_valid [1]) for a token stream split across data-parallel ranks.

    Each rank passes its own contiguous range of the stream, ranges in rank order and every
    range but the last a multiple of 1024 tokens.  w is this rank's; D3 and n_valid are the
    whole stream's, with the bits of one ``importance_weights`` call over it (the block
    partials are gathered, then every rank runs the same fixed tree).
    """
    import torch.distributed as dist

    T = int(logp_pi.shape[0])
    rank, world = dist.get_rank(group), dist.get_world_size(group)
    if rank < world - 1 and T % IS_BLOCK != 0:
        raise ValueError(f"rank {rank} holds {T} tokens: every rank but the last must hold a "
                         f"multiple of {IS_BLOCK}")
    w, blk_sum, blk_cnt = engine.importance_weights_partials(logp_pi, logp_mu, mask)
    all_sum, all_cnt = gather_block_partials(blk_sum, blk_cnt, group=group)
    d3, n_valid = engine.d3_from_partials(all_sum, all_cnt)
    return w, d3, n_valid


def acceptance_stats_data_parallel(engine: "Engine", logp_a: torch.Tensor, logp_b: torch.Tensor,
                                   mask: torch.Tensor = None, group=None):
    """fp64 [5] acceptance statistics of a token stream split across data-parallel ranks,
    under the same rules as ``importance_weights_data_parallel``; bit-identical to one
    ``acceptance_stats`` call over the whole stream."""
    import torch.distributed as dist

    T = int(logp_a.shape[0])
    rank, world = dist.get_rank(group), dist.get_world_size(group)
    if rank < world - 1 and T % IS_BLOCK != 0:
        raise ValueError(f"rank {rank} holds {T} tokens: every rank but the last must hold a "
                         f"multiple of {IS_BLOCK}")
    sums, bmax, cnts = engine.acceptance_stats_partials(logp_a, logp_b, mask)
    all_sums, all_max, all_cnts = gather_block_partials(sums, bmax, cnts, group=group)
    return engine.acceptance_stats_from_partials(all_sums, all_max, all_cnts)


def gather_vocab_partials(ms: torch.Tensor, zy: torch.Tensor, ids: torch.Tensor, v0: int,
                          V_local: int, V_full: int, group=None):
    """The exchange of a vocabulary-parallel logprob: every rank's tile partials ms
    [tiles, T, 2] all-gathered in vocabulary order, and each row's sampled logit taken from
    the rank whose slice [v0, v0 + V_local) holds its (global) id.  Data movement only.
    Returns (ms_all [ceil(V_full/64), T, 2], zy_all [T])."""
    import torch.distributed as dist

    if v0 % 128 != 0:
        raise ValueError(f"a vocabulary slice must start at a multiple of 128 rows (got {v0})")
    world = dist.get_world_size(group)
    bounds = torch.tensor([v0, V_local], dtype=torch.int64, device=ms.device)
    all_bounds = [torch.empty_like(bounds) for _ in range(world)]
    dist.all_gather(all_bounds, bounds, group=group)
    starts = [int(b[0]) for b in all_bounds]
    ends = [int(b[0] + b[1]) for b in all_bounds]
    if starts[0] != 0 or ends[-1] != V_full or any(e != s for e, s in zip(ends[:-1], starts[1:])):
        raise ValueError("the slices must cover [0, V_full) in rank order")
    (ms_t,) = gather_block_partials(ms.permute(1, 2, 0).contiguous(), group=group)
    ms_all = ms_t.permute(2, 0, 1).contiguous()
    zys = [torch.empty_like(zy) for _ in range(world)]
    dist.all_gather(zys, zy.contiguous(), group=group)
    start_t = torch.tensor(starts, dtype=torch.int64, device=ms.device)
    owner = (torch.searchsorted(start_t, ids.to(torch.int64), right=True) - 1).clamp_(0, world - 1)
    zy_all = torch.stack(zys)[owner, torch.arange(zy.shape[0], device=ms.device)].contiguous()
    return ms_all, zy_all


def logprobs_vocab_parallel(engine: "Engine", X: torch.Tensor, ids: torch.Tensor, v0: int,
                            V_full: int, return_logZ: bool = False, group=None):
    """Sampled-token logprobs with the lm_head split by vocabulary across ranks.

    ``engine`` is this rank's handle over the rows [v0, v0 + engine.V) of the full lm_head;
    ranks hold consecutive slices in rank order, each starting at a multiple of 128 rows.
    Every rank passes the same X and (global) ids and gets the full-vocabulary logp, with the
    bits of one ``logprobs`` call on the whole lm_head (``gather_vocab_partials`` moves the
    partials; the fixed tile tree finishes them).
    """
    if v0 % 128 != 0:
        raise ValueError(f"a vocabulary slice must start at a multiple of 128 rows (got {v0})")
    ms, zy = engine.vocab_partials(X, ids - v0)
    ms_all, zy_all = gather_vocab_partials(ms, zy, ids, v0, engine.V, V_full, group)
    return engine.logprobs_from_vocab_partials(V_full, ms_all, zy_all, ids,
                                               return_logZ=return_logZ)
