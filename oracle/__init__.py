"""CPU oracle (fp64) for the sampled-token logprob path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  The product path (``bit_consistent_logprob_gb300``)
never imports it and has no CPU fallback.  The arithmetic lives in
``oracle/oracle.c`` (plain C, fp64, OpenMP over rows); this module only builds
it with gcc and marshals numpy arrays through ctypes.

Functions and the passages they follow are listed in the header of
``oracle.c``.  Parity status: every function is pinned by the ``not gpu`` tests
in ``tests/test_oracle.py`` (exact rational arithmetic, closed forms, golden
values under ``tests/golden/``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_CFLAGS = ["-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-std=c11"]


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (gcc, no -march flags)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, i32 = ctypes.c_int64, ctypes.c_int32
        p = ctypes.c_void_p
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_logits.argtypes = [p, i64, p, i64, i64, p, i64, p]
        lib.oracle_logprobs.argtypes = [p, i64, p, p, i64, i64, p, i64, p, p]
        lib.oracle_log_softmax.argtypes = [p, i64, p, i64, i64, p, i64, p]
        lib.oracle_leaf_sums.argtypes = [p, p, i64, i32, p]
        lib.oracle_tree_fp32.argtypes = [p, i32]
        lib.oracle_tree_fp32.restype = ctypes.c_float
        lib.oracle_tree_fp32_many.argtypes = [p, i32, i64, p]
        lib.oracle_acceptance_stats.argtypes = [p, p, p, i64, p]
        lib.oracle_entropy.argtypes = [p, i64, p, i64, i64, p, i64, p]
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_quantize_blocks.argtypes = [p, i64, i64, i64, i64, p, p]
        lib.oracle_logprobs_fp8.argtypes = [p, p, p, p, p, i64, i64, p, i64, p, p]
        lib.oracle_entropy_fp8.argtypes = [p, p, p, p, i64, i64, p, i64, p]
        lib.oracle_logprobs_f64.argtypes = [p, p, p, i64, i64, i64, p]
        lib.oracle_logprob_grad.argtypes = [p, p, p, p, i64, i64, i64, p, p, p]
        lib.oracle_reinforce_zero.argtypes = [p, p, p, p, i64, p, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_double, ctypes.c_float, ctypes.c_float,
                                              ctypes.c_double, ctypes.c_double,
                                              p, p, p, p, p, p]
        lib.oracle_importance_weights.argtypes = [p, p, p, i64, p, p, p, p]
        for f in (lib.oracle_logits, lib.oracle_logprobs, lib.oracle_log_softmax,
                  lib.oracle_leaf_sums, lib.oracle_tree_fp32_many,
                  lib.oracle_importance_weights):
            f.restype = None
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> ctypes.c_void_p:
    return ctypes.c_void_p(a.ctypes.data)


def _u16_2d(a) -> np.ndarray:
    """Accept a numpy uint16/int16 array or a torch bf16 tensor; return uint16 [rows, cols]."""
    if hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        import torch  # local: only the bf16 view needs torch

        a = a.detach().to("cpu").contiguous().view(torch.int16).numpy()
    a = np.asarray(a)
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16 or a.ndim != 2:
        raise TypeError("expected a 2-D bf16 bit array")
    return a


def _rows_arg(rows, T: int) -> np.ndarray:
    if rows is None:
        return np.arange(T, dtype=np.int64)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    if rows.size and (rows.min() < 0 or rows.max() >= T):
        raise IndexError("row index out of range")
    return rows


def num_threads() -> int:
    """Number of OpenMP threads the oracle uses."""
    return int(_load().oracle_num_threads())


def logits(X, W, rows=None) -> np.ndarray:
    """fp64 logits z[r, v] = sum_k X[rows[r], k] W[v, k]."""
    X, W = _u16_2d(X), _u16_2d(W)
    Xc = np.ascontiguousarray(X)
    Wc = np.ascontiguousarray(W)
    T, H = Xc.shape
    V = Wc.shape[0]
    assert Wc.shape[1] == H
    r = _rows_arg(rows, T)
    out = np.empty((r.size, V), dtype=np.float64)
    _load().oracle_logits(_ptr(Xc), H, _ptr(Wc), H, V, _ptr(r), r.size, _ptr(out))
    return out


def logprobs(X, W, ids, rows=None):
    """Sampled-token logprob and log-partition for the listed rows (fp64).

    Returns (logp[nrows], logZ[nrows]).  ids is indexed by row number."""
    X, W = _u16_2d(X), _u16_2d(W)
    Xc = np.ascontiguousarray(X)
    Wc = np.ascontiguousarray(W)
    T, H = Xc.shape
    V = Wc.shape[0]
    assert Wc.shape[1] == H
    ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    assert ids.shape == (T,)
    r = _rows_arg(rows, T)
    logp = np.empty(r.size, dtype=np.float64)
    logZ = np.empty(r.size, dtype=np.float64)
    _load().oracle_logprobs(_ptr(Xc), H, _ptr(Wc), _ptr(ids), H, V, _ptr(r), r.size,
                            _ptr(logp), _ptr(logZ))
    return logp, logZ


def log_softmax(X, W, rows=None) -> np.ndarray:
    """Full fp64 log-softmax over the vocabulary for the listed rows: [nrows, V]."""
    X, W = _u16_2d(X), _u16_2d(W)
    Xc = np.ascontiguousarray(X)
    Wc = np.ascontiguousarray(W)
    T, H = Xc.shape
    V = Wc.shape[0]
    r = _rows_arg(rows, T)
    out = np.empty((r.size, V), dtype=np.float64)
    _load().oracle_log_softmax(_ptr(Xc), H, _ptr(Wc), H, V, _ptr(r), r.size, _ptr(out))
    return out


def leaf_sums(xrow, wrow, n_leaves: int) -> np.ndarray:
    """fp64 sums over each of the n_leaves contiguous K leaves of one (row, vocab) pair."""
    x = _u16_2d(xrow.reshape(1, -1))[0]
    w = _u16_2d(wrow.reshape(1, -1))[0]
    H = x.shape[0]
    if H % n_leaves or w.shape[0] != H:
        raise ValueError("H must be a multiple of n_leaves and the rows must match")
    out = np.empty(n_leaves, dtype=np.float64)
    xc, wc = np.ascontiguousarray(x), np.ascontiguousarray(w)
    _load().oracle_leaf_sums(_ptr(xc), _ptr(wc), H, n_leaves, _ptr(out))
    return out


def tree_fp32(P) -> np.ndarray:
    """Fixed pairwise fp32 tree over the last axis of P ([..., N], N a power of two)."""
    P = np.ascontiguousarray(np.asarray(P, dtype=np.float32))
    N = P.shape[-1]
    flat = P.reshape(-1, N)
    out = np.empty(flat.shape[0], dtype=np.float32)
    _load().oracle_tree_fp32_many(_ptr(flat), N, flat.shape[0], _ptr(out))
    return out.reshape(P.shape[:-1])


def importance_weights(logp_pi, logp_mu, mask=None):
    """w = exp(log pi - log mu), term = w - 1 - log w, D3 = mean term over valid tokens.

    Returns (w f64[T], term f64[T], d3 float, n_valid int)."""
    a = np.ascontiguousarray(np.asarray(logp_pi, dtype=np.float32))
    b = np.ascontiguousarray(np.asarray(logp_mu, dtype=np.float32))
    assert a.shape == b.shape and a.ndim == 1
    T = a.size
    m = None
    if mask is not None:
        m = np.ascontiguousarray(np.asarray(mask).astype(np.uint8))
        assert m.shape == (T,)
    w = np.empty(T, dtype=np.float64)
    term = np.empty(T, dtype=np.float64)
    d3 = np.zeros(1, dtype=np.float64)
    nv = np.zeros(1, dtype=np.int64)
    _load().oracle_importance_weights(_ptr(a), _ptr(b), None if m is None else _ptr(m), T,
                                      _ptr(w), _ptr(term), _ptr(d3), _ptr(nv))
    return w, term, float(d3[0]), int(nv[0])


def _f32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _mask_arg(mask, T):
    if mask is None:
        return None
    m = np.ascontiguousarray(np.asarray(mask).astype(np.uint8))
    assert m.shape == (T,)
    return m


def acceptance_stats(logp_a, logp_b, mask=None) -> dict:
    """max, mean, std (population) of |a - b| and k3 = mean(r - 1 - log r), r = e^(a-b),
    over valid tokens; n_valid."""
    a, b = _f32(logp_a), _f32(logp_b)
    assert a.shape == b.shape and a.ndim == 1
    m = _mask_arg(mask, a.size)
    out = np.zeros(5, dtype=np.float64)
    _load().oracle_acceptance_stats(_ptr(a), _ptr(b), None if m is None else _ptr(m), a.size,
                                    _ptr(out))
    return dict(max=out[0], mean=out[1], std=out[2], k3=out[3], n_valid=int(out[4]))


TIS, TOKEN_GATE, SEQ_GATE = 1, 2, 4


def reinforce_zero(logp_pi, logp_mu, offsets, rewards, group_size, mask=None, flags=0,
                   tis_cap=float("inf"), token_log_lo=-float("inf"),
                   token_log_hi=float("inf"), seq_log_lo=-float("inf"),
                   seq_log_hi=float("inf")) -> dict:
    """REINFORCE Zero loss, weights and dL/dlog pi for responses packed at ``offsets``.

    Returns dict(loss, w_hat[T], grad[T], adv[B], seq_logratio[B], kept[B]) in fp64."""
    a, b = _f32(logp_pi), _f32(logp_mu)
    T = a.size
    offs = np.ascontiguousarray(np.asarray(offsets, dtype=np.int64))
    B = offs.size - 1
    assert B >= 0 and offs[0] == 0 and offs[-1] == T and np.all(np.diff(offs) >= 0)
    r = _f32(rewards)
    assert r.shape == (B,) and group_size >= 1 and B % group_size == 0
    m = _mask_arg(mask, T)
    w_hat = np.zeros(T, dtype=np.float64)
    grad = np.zeros(T, dtype=np.float64)
    adv = np.zeros(B, dtype=np.float64)
    slr = np.zeros(B, dtype=np.float64)
    kept = np.zeros(B, dtype=np.int32)
    loss = np.zeros(1, dtype=np.float64)
    _load().oracle_reinforce_zero(_ptr(a), _ptr(b), None if m is None else _ptr(m), _ptr(offs), B,
                                  _ptr(r), int(group_size), int(flags), float(tis_cap),
                                  float(token_log_lo), float(token_log_hi), float(seq_log_lo),
                                  float(seq_log_hi), _ptr(w_hat), _ptr(grad), _ptr(adv), _ptr(slr),
                                  _ptr(kept), _ptr(loss))
    return dict(loss=float(loss[0]), w_hat=w_hat, grad=grad, adv=adv, seq_logratio=slr,
                kept=kept.astype(bool))


def entropy(X, W, rows=None) -> np.ndarray:
    """Softmax entropy -sum_v p log p of the listed rows (fp64)."""
    X, W = _u16_2d(X), _u16_2d(W)
    Xc, Wc = np.ascontiguousarray(X), np.ascontiguousarray(W)
    T, H = Xc.shape
    V = Wc.shape[0]
    r = _rows_arg(rows, T)
    out = np.empty(r.size, dtype=np.float64)
    _load().oracle_entropy(_ptr(Xc), H, _ptr(Wc), H, V, _ptr(r), r.size, _ptr(out))
    return out


def logprobs_f64(X, W, ids) -> np.ndarray:
    """Sampled-token logprobs of real-valued (fp64) X [T, H] and W [V, H]."""
    Xd = np.ascontiguousarray(np.asarray(X, dtype=np.float64))
    Wd = np.ascontiguousarray(np.asarray(W, dtype=np.float64))
    T, H = Xd.shape
    V = Wd.shape[0]
    ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    out = np.empty(T, dtype=np.float64)
    _load().oracle_logprobs_f64(_ptr(Xd), _ptr(Wd), _ptr(ids), T, H, V, _ptr(out))
    return out


def logprob_grad(X, W, ids, g):
    """Gradient of sum_t g_t logp_t: returns (dX [T,H], dW [V,H], dl [T,V]) in fp64."""
    X, W = _u16_2d(X), _u16_2d(W)
    Xc, Wc = np.ascontiguousarray(X), np.ascontiguousarray(W)
    T, H = Xc.shape
    V = Wc.shape[0]
    ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    g = np.ascontiguousarray(np.asarray(g, dtype=np.float64))
    assert ids.shape == (T,) and g.shape == (T,)
    dX = np.empty((T, H), dtype=np.float64)
    dW = np.empty((V, H), dtype=np.float64)
    dl = np.empty((T, V), dtype=np.float64)
    _load().oracle_logprob_grad(_ptr(Xc), _ptr(Wc), _ptr(ids), _ptr(g), T, H, V, _ptr(dX),
                                _ptr(dW), _ptr(dl))
    return dX, dW, dl


def e4m3_decode(codes) -> np.ndarray:
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([lib.oracle_e4m3_decode(int(v)) for v in c], dtype=np.float64)


def e4m3_encode(values) -> np.ndarray:
    lib = _load()
    x = np.asarray(values, dtype=np.float32).ravel()
    return np.array([lib.oracle_e4m3_encode(float(v)) for v in x], dtype=np.uint8)


def quantize_blocks(M, block_rows: int):
    """Block-FP8 quantisation of a bf16 matrix [rows, cols]: (q uint8 [rows, cols],
    scales float32 [ceil(rows / block_rows), cols / 128])."""
    M = np.ascontiguousarray(_u16_2d(M))
    rows, cols = M.shape
    assert cols % 128 == 0
    q = np.empty((rows, cols), dtype=np.uint8)
    scales = np.empty(((rows + block_rows - 1) // block_rows, cols // 128), dtype=np.float32)
    _load().oracle_quantize_blocks(_ptr(M), rows, cols, cols, block_rows, _ptr(q), _ptr(scales))
    return q, scales


def logprobs_fp8(xq, sx, wq, sw, ids, rows=None):
    """Sampled-token logprob and logZ (fp64) from block-FP8 operands."""
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    sx = np.ascontiguousarray(sx, dtype=np.float32)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    T, H = xq.shape
    V = wq.shape[0]
    ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
    r = _rows_arg(rows, T)
    logp = np.empty(r.size, dtype=np.float64)
    logZ = np.empty(r.size, dtype=np.float64)
    _load().oracle_logprobs_fp8(_ptr(xq), _ptr(sx), _ptr(wq), _ptr(sw), _ptr(ids), H, V, _ptr(r),
                                r.size, _ptr(logp), _ptr(logZ))
    return logp, logZ


def entropy_fp8(xq, sx, wq, sw, rows=None) -> np.ndarray:
    """Softmax entropy (fp64) of the listed rows, logits from block-FP8 operands."""
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    sx = np.ascontiguousarray(sx, dtype=np.float32)
    sw = np.ascontiguousarray(sw, dtype=np.float32)
    T, H = xq.shape
    V = wq.shape[0]
    r = _rows_arg(rows, T)
    out = np.empty(r.size, dtype=np.float64)
    _load().oracle_entropy_fp8(_ptr(xq), _ptr(sx), _ptr(wq), _ptr(sw), H, V, _ptr(r), r.size,
                               _ptr(out))
    return out
