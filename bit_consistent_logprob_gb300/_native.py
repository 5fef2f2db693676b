"""ctypes binding of ``liblp.so`` (the C ABI in ``include/lp.h``).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind these entry points.  There is no fallback: if the library has
not been built, loading fails with an error that says how to build it.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

LP_OK, LP_ERR_INVALID_ARG, LP_ERR_UNSUPPORTED, LP_ERR_CUDA, LP_ERR_OOM, LP_ERR_TIMEOUT = range(6)
STATUS_NAMES = {
    LP_OK: "LP_OK", LP_ERR_INVALID_ARG: "LP_ERR_INVALID_ARG",
    LP_ERR_UNSUPPORTED: "LP_ERR_UNSUPPORTED", LP_ERR_CUDA: "LP_ERR_CUDA",
    LP_ERR_OOM: "LP_ERR_OOM", LP_ERR_TIMEOUT: "LP_ERR_TIMEOUT",
}
LP_PHASE_AUTO, LP_PHASE_PREFILL, LP_PHASE_DECODE = 0, 1, 2
LP_PROFILE_LEAF_GEMM, LP_PROFILE_GRAD_DX, LP_PROFILE_GRAD_DW = 0, 1, 2

# Every symbol include/lp.h declares, with its ctypes signature.
_p = ctypes.c_void_p
_i32, _i64 = ctypes.c_int32, ctypes.c_int64


class LpConfig(ctypes.Structure):
    _fields_ = [("H", ctypes.c_int32), ("V", ctypes.c_int32), ("n_leaves", ctypes.c_int32),
                ("tp_slices", ctypes.c_int32), ("max_tokens", ctypes.c_int64)]


class LpRzOptions(ctypes.Structure):
    _fields_ = [("flags", ctypes.c_int32), ("tis_cap", ctypes.c_float),
                ("token_log_lo", ctypes.c_float), ("token_log_hi", ctypes.c_float),
                ("seq_log_lo", ctypes.c_double), ("seq_log_hi", ctypes.c_double)]


LP_RZ_TIS, LP_RZ_TOKEN_GATE, LP_RZ_SEQ_GATE = 1, 2, 4
LP_STAT_MAX_ABS, LP_STAT_MEAN_ABS, LP_STAT_STD_ABS, LP_STAT_K3, LP_STAT_N_VALID = range(5)
LP_STAT_COUNT = 5

SIGNATURES = {
    "lp_init": (ctypes.c_int, [ctypes.POINTER(LpConfig), _p, _p, ctypes.POINTER(_p)]),
    "lp_logprobs": (ctypes.c_int, [_p, _p, _i64, _p, _i64, _p, _p, ctypes.c_int, _p]),
    "lp_logprobs_host": (ctypes.c_int, [_p, _p, _i64, _p, _i64, _p, _p, _p]),
    "lp_logits_partial": (ctypes.c_int, [_p, _p, _i64, _i64, _i32, _i32, _p, _i64, _p]),
    "lp_logprobs_from_partials": (ctypes.c_int, [_p, _p, _i32, _i64, _i64, _p, _i64, _p, _p, _p]),
    "lp_importance_weights": (ctypes.c_int, [_p, _p, _p, _p, _i64, _p, _p, _p, _p]),
    "lp_importance_weights_host": (ctypes.c_int, [_p, _p, _p, _p, _i64, _p, _p, _p, _p]),
    "lp_importance_weights_partials": (ctypes.c_int, [_p, _p, _p, _p, _i64, _p, _p, _p, _p]),
    "lp_d3_from_partials": (ctypes.c_int, [_p, _p, _p, _i64, _p, _p, _p]),
    "lp_vocab_partials": (ctypes.c_int, [_p, _p, _i64, _p, _i64, _p, _i64, _p, _p]),
    "lp_logprobs_from_vocab_partials": (ctypes.c_int, [_p, _i32, _p, _i64, _p, _p, _i64, _p, _p,
                                                       _p]),
    "lp_acceptance_stats_partials": (ctypes.c_int, [_p, _p, _p, _p, _i64, _p, _p, _p, _p]),
    "lp_acceptance_stats_from_partials": (ctypes.c_int, [_p, _p, _p, _p, _i64, _p, _p]),
    "lp_acceptance_stats": (ctypes.c_int, [_p, _p, _p, _p, _i64, _p, _p]),
    "lp_logprobs_entropy": (ctypes.c_int, [_p, _p, _i64, _p, _i64, _p, _p, _p, ctypes.c_int, _p]),
    "lp_logprobs_backward": (ctypes.c_int, [_p, _p, _i64, _p, _p, _p, _i64, _p, _p, ctypes.c_int,
                                            _p]),
    "lp_backward_reserve": (ctypes.c_int, [_p, _i64]),
    "lp_init_fp8": (ctypes.c_int, [ctypes.POINTER(LpConfig), _p, _p, ctypes.POINTER(_p)]),
    "lp_fp8_requantize": (ctypes.c_int, [_p, _p]),
    "lp_fp8_weights": (ctypes.c_int, [_p, ctypes.POINTER(_p), ctypes.POINTER(_p)]),
    "lp_fp8_quantize_x": (ctypes.c_int, [_p, _p, _i64, _i64, _p, _p, _p]),
    "lp_contract": (ctypes.c_int, [ctypes.POINTER(LpConfig), ctypes.c_int, _p, ctypes.c_size_t,
                                   ctypes.POINTER(ctypes.c_size_t)]),
    "lp_contract_digest": (ctypes.c_int, [ctypes.POINTER(LpConfig), ctypes.c_int, ctypes.c_int,
                                          _p]),
    "lp_contract_check": (ctypes.c_int, [ctypes.POINTER(LpConfig), ctypes.c_int, _p, _p]),
    "lp_sha256": (None, [_p, ctypes.c_size_t, _p]),
    "lp_reinforce_zero": (ctypes.c_int, [_p, _p, _p, _p, _i64, _p, _i64, _p, _i32,
                                         ctypes.POINTER(LpRzOptions), _p, _p, _p, _p, _p, _p]),
    "lp_profile_enable": (ctypes.c_int, [_p, ctypes.c_int]),
    "lp_profile_read": (ctypes.c_int, [_p, ctypes.POINTER(ctypes.c_double),
                                       ctypes.POINTER(ctypes.c_int32)]),
    "lp_profile_read_kind": (ctypes.c_int, [_p, ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                                            ctypes.POINTER(ctypes.c_int32)]),
    "lp_logprobs_noalloc": (ctypes.c_int, [_p, _i32, _i32, _i32, _p, _i64, _p, _i64, _p, _p, _p]),
    "lp_noalloc_last_error": (ctypes.c_char_p, []),
    "lp_check": (ctypes.c_int, [_p]),
    "lp_selftest_wait_timeout": (ctypes.c_int, [_p, _i64, _p]),
    "lp_clear_status": (ctypes.c_int, [_p, _p]),
    "lp_last_error": (ctypes.c_char_p, []),
    "lp_workspace_bytes": (ctypes.c_int64, [_p]),
    "lp_last_launch_count": (ctypes.c_int32, [_p]),
    "lp_version": (ctypes.c_int, []),
    "lp_free": (None, [_p]),
}


class LpError(RuntimeError):
    """A non-zero lp_status returned by the native library."""

    def __init__(self, code: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {message}")
        self.code = code


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = False):
    """Load liblp.so (optionally building it first).  Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIB_PATH
        if build_if_missing:
            path = _build.build()
        if not os.path.exists(path):
            raise RuntimeError(
                f"native library {path} is missing; build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` "
                "(there is no CPU or PyTorch fallback)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def check(rc: int) -> None:
    if rc != LP_OK:
        msg = load().lp_last_error()
        raise LpError(rc, msg.decode() if msg else "")
