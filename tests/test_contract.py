"""The execution contract and its SHA-256 identities (host code; runs without a GPU).

IsoExec's contract (SkyRL blog summary, "unified execution contract") identifies the
numerics two runtimes share by SHA-256 digests of the serialised contract.  Checks: the
library's SHA-256 against Python's hashlib (FIPS 180-4 test lengths around the padding
boundaries), the identities against hashlib over the canonical sections (so a third party
can recompute them from the published JSON), which settings move which digest, and the
peer check.
"""
import hashlib
import json
import os

import pytest

from bit_consistent_logprob_gb300 import LpError, contract, _native


@pytest.fixture(scope="module", autouse=True)
def lib():
    return _native.load(build_if_missing=True)


@pytest.mark.parametrize("n", [0, 1, 3, 55, 56, 63, 64, 65, 119, 120, 127, 128, 1000, 1 << 20])
def test_sha256_matches_hashlib(n):
    data = bytes((i * 131 + 7) & 0xFF for i in range(n)) if n < 5000 else os.urandom(n)
    assert contract.sha256(data) == hashlib.sha256(data).digest()


def test_sha256_known_vector():
    assert contract.sha256(b"abc").hex() == hashlib.sha256(b"abc").hexdigest()


def test_identities_are_sha256_of_the_canonical_sections():
    doc = contract.contract(H=7168, V=129280, n_leaves=8, tp_slices=2, max_tokens=2048)
    for key in ("semantic", "numerical_policy", "deployment"):
        canon = json.dumps(doc[key], separators=(",", ":")).encode()
        assert doc["identities"][key] == hashlib.sha256(canon).hexdigest(), key
    assert doc["numerical_policy"]["composition"][0]["constants"]["leaves"] == 8
    assert doc["numerical_policy"]["composition"][0]["constants"]["leaf_dtype"] == "fp32"
    assert doc["numerical_policy"]["claims"]["topology"]["tp_slices"] == [1, 2, 4, 8]
    raw = contract.contract_json(H=7168, V=129280)
    assert raw == contract.contract_json(H=7168, V=129280)  # deterministic


def test_which_settings_move_which_digest():
    d = lambda w, **kw: contract.digest(w, **{**dict(H=2048, V=151936), **kw})  # noqa: E731
    pol = contract.NUMERICAL_POLICY
    # row chunking and the emulated TP split are proven not to change bits
    assert d(pol) == d(pol, max_tokens=7) == d(pol, tp_slices=4)
    assert d(contract.DEPLOYMENT) != d(contract.DEPLOYMENT, max_tokens=7)
    # the leaf count is a pinned constant; the shape is part of the semantics
    assert d(pol) != d(pol, n_leaves=4)
    assert d(contract.SEMANTIC) != d(contract.SEMANTIC, V=151937)
    assert d(contract.SEMANTIC) == d(contract.SEMANTIC, n_leaves=4)


def test_block_fp8_policy_differs_and_is_canonical():
    kw = dict(H=7168, V=129280)
    doc = contract.contract(precision=contract.FP8_BLOCK, **kw)
    for key in ("semantic", "numerical_policy", "deployment"):
        canon = json.dumps(doc[key], separators=(",", ":")).encode()
        assert doc["identities"][key] == hashlib.sha256(canon).hexdigest(), key
    lm = doc["numerical_policy"]["composition"][0]
    assert lm["constants"]["input_dtype"] == "e4m3"
    assert lm["constants"]["quantization"]["weight_block"] == "128x128"
    assert doc["numerical_policy"]["claims"]["topology"]["tp_slices"] == [1, 2, 4, 8]
    contract.contract(precision=contract.FP8_BLOCK, tp_slices=4, **kw)  # a proven split
    pol = contract.NUMERICAL_POLICY
    assert contract.digest(pol, precision=contract.FP8_BLOCK, **kw) != contract.digest(pol, **kw)
    assert (contract.digest(contract.SEMANTIC, precision=contract.FP8_BLOCK, **kw)
            == contract.digest(contract.SEMANTIC, **kw))
    with pytest.raises(LpError):
        contract.digest(pol, precision=contract.FP8_BLOCK, H=512, V=1000, n_leaves=8)


def test_peer_check():
    kw = dict(H=2048, V=151936)
    sem, pol = contract.digest(contract.SEMANTIC, **kw), contract.digest(contract.NUMERICAL_POLICY, **kw)
    contract.check_peer(sem, pol, max_tokens=99, **kw)  # deployment may differ
    other = contract.digest(contract.NUMERICAL_POLICY, n_leaves=4, **kw)
    with pytest.raises(LpError, match="numerical_policy"):
        contract.check_peer(sem, other, **kw)
    with pytest.raises(LpError):
        contract.digest(contract.SEMANTIC, H=100, V=10)  # H not a multiple of 64 * leaves
