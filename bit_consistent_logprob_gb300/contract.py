"""Execution contract of a configuration (``lp_contract`` in ``include/lp.h``).

Host-only calls into ``liblp.so``: no device and no handle are needed, so a trainer and a
rollout engine can exchange and compare the digests before either runs a kernel.
"""
from __future__ import annotations

import ctypes
import json

from . import _native

SEMANTIC, NUMERICAL_POLICY, DEPLOYMENT = 0, 1, 2
BF16, FP8_BLOCK = 0, 1


def _cfg(H, V, n_leaves, tp_slices, max_tokens):
    return _native.LpConfig(int(H), int(V), int(n_leaves), int(tp_slices), int(max_tokens))


def contract_json(H: int, V: int, n_leaves: int = 8, tp_slices: int = 1,
                  max_tokens: int = 16384, precision: int = BF16) -> str:
    """The canonical contract JSON (with its SHA-256 identities) as a string."""
    lib = _native.load()
    cfg = _cfg(H, V, n_leaves, tp_slices, max_tokens)
    n = ctypes.c_size_t()
    _native.check(lib.lp_contract(ctypes.byref(cfg), int(precision), None, 0, ctypes.byref(n)))
    buf = ctypes.create_string_buffer(n.value + 1)
    _native.check(lib.lp_contract(ctypes.byref(cfg), int(precision), buf, n.value + 1,
                                  ctypes.byref(n)))
    return buf.value.decode()


def contract(H: int, V: int, n_leaves: int = 8, tp_slices: int = 1,
             max_tokens: int = 16384, precision: int = BF16) -> dict:
    return json.loads(contract_json(H, V, n_leaves, tp_slices, max_tokens, precision))


def digest(which: int, H: int, V: int, n_leaves: int = 8, tp_slices: int = 1,
           max_tokens: int = 16384, precision: int = BF16) -> bytes:
    lib = _native.load()
    cfg = _cfg(H, V, n_leaves, tp_slices, max_tokens)
    out = (ctypes.c_uint8 * 32)()
    _native.check(lib.lp_contract_digest(ctypes.byref(cfg), int(precision), int(which), out))
    return bytes(out)


def check_peer(peer_semantic: bytes, peer_numerical_policy: bytes, H: int, V: int,
               n_leaves: int = 8, tp_slices: int = 1, max_tokens: int = 16384,
               precision: int = BF16) -> None:
    """Raise LpError unless the peer's semantic and numerical-policy digests match ours."""
    lib = _native.load()
    cfg = _cfg(H, V, n_leaves, tp_slices, max_tokens)
    a = (ctypes.c_uint8 * 32).from_buffer_copy(peer_semantic)
    b = (ctypes.c_uint8 * 32).from_buffer_copy(peer_numerical_policy)
    _native.check(lib.lp_contract_check(ctypes.byref(cfg), int(precision), a, b))


def sha256(data: bytes) -> bytes:
    """The library's own SHA-256 (exported for verification)."""
    out = (ctypes.c_uint8 * 32)()
    _native.load().lp_sha256(data, len(data), out)
    return bytes(out)
