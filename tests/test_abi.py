"""C ABI checks that need no GPU: the library builds, loads and exports every symbol
include/lp.h declares, and host-side argument validation answers before any CUDA call."""
import ctypes
import os
import re

import pytest

from bit_consistent_logprob_gb300 import _native
from bit_consistent_logprob_gb300._native import (LP_ERR_INVALID_ARG, LP_ERR_UNSUPPORTED, LP_OK,
                                                  LpConfig)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    return _native.load(build_if_missing=True)


def declared_functions():
    text = open(os.path.join(ROOT, "include", "lp.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*LP_API\s+(?:const\s+)?[\w]+\s*\*?\s*(lp_\w+)\s*\(", text,
                       flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("lp_init", "lp_logprobs", "lp_importance_weights", "lp_free", "lp_check",
                     "lp_last_error", "lp_logits_partial", "lp_logprobs_from_partials",
                     "lp_logprobs_host"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _native.SIGNATURES, f"binding lacks a signature for {name}"


def test_binding_declares_nothing_the_header_lacks():
    assert set(_native.SIGNATURES) <= set(declared_functions())


def test_version_and_error_string(lib):
    assert lib.lp_version() == 100
    assert isinstance(lib.lp_last_error(), bytes)


def _init(lib, H=256, V=4096, N=4, s=1, max_tokens=64, W=0x10000):
    cfg = LpConfig(H, V, N, s, max_tokens)
    h = ctypes.c_void_p()
    rc = lib.lp_init(ctypes.byref(cfg), ctypes.c_void_p(W), None, ctypes.byref(h))
    return rc, h


@pytest.mark.parametrize("kwargs,code", [
    (dict(N=3), LP_ERR_UNSUPPORTED),            # leaves must be a power of two
    (dict(N=16), LP_ERR_UNSUPPORTED),           # outside the proven set
    (dict(H=200), LP_ERR_UNSUPPORTED),          # leaf length not a multiple of 64
    (dict(H=256, N=8), LP_ERR_UNSUPPORTED),     # 32-element leaves
    (dict(s=3), LP_ERR_UNSUPPORTED),            # TP split not a power of two
    (dict(N=4, s=8), LP_ERR_UNSUPPORTED),       # TP split must divide the leaves
    (dict(max_tokens=0), LP_ERR_INVALID_ARG),
    (dict(V=0), LP_ERR_INVALID_ARG),
    (dict(W=0), LP_ERR_INVALID_ARG),            # NULL weights
    (dict(W=0x10008), LP_ERR_INVALID_ARG),      # weights not 16-byte aligned
])
def test_init_rejects_before_touching_the_device(lib, kwargs, code):
    rc, h = _init(lib, **kwargs)
    assert rc == code
    assert not h.value
    assert lib.lp_last_error()


def test_null_handle_is_rejected(lib):
    assert lib.lp_logprobs(None, None, 256, None, 0, None, None, 0, None) == LP_ERR_INVALID_ARG
    assert lib.lp_importance_weights(None, None, None, None, 0, None, None, None,
                                     None) == LP_ERR_INVALID_ARG
    assert lib.lp_check(None) == LP_ERR_INVALID_ARG
    assert lib.lp_logits_partial(None, None, 256, 0, 0, 1, None, 0, None) == LP_ERR_INVALID_ARG
    lib.lp_free(None)  # no-op
    assert lib.lp_workspace_bytes(None) == 0
    assert LP_OK == 0


def test_null_handle_is_rejected_by_the_parallel_exchange_calls(lib):
    # the partial-export and finish calls of the data- and vocabulary-parallel splits
    # validate on the host before any CUDA call
    assert lib.lp_importance_weights_partials(None, None, None, None, 0, None, None, None,
                                              None) == LP_ERR_INVALID_ARG
    assert lib.lp_d3_from_partials(None, None, None, 0, None, None, None) == LP_ERR_INVALID_ARG
    assert lib.lp_acceptance_stats_partials(None, None, None, None, 0, None, None, None,
                                            None) == LP_ERR_INVALID_ARG
    assert lib.lp_acceptance_stats_from_partials(None, None, None, None, 0, None,
                                                 None) == LP_ERR_INVALID_ARG
    assert lib.lp_vocab_partials(None, None, 256, None, 0, None, 0, None,
                                 None) == LP_ERR_INVALID_ARG
    assert lib.lp_logprobs_from_vocab_partials(None, 4096, None, 0, None, None, 0, None, None,
                                               None) == LP_ERR_INVALID_ARG


def test_block_size_of_the_header_and_the_binding_agree():
    import re

    from bit_consistent_logprob_gb300.engine import IS_BLOCK

    with open(os.path.join(ROOT, "include", "lp.h")) as f:
        m = re.search(r"#define LP_IS_BLOCK (\d+)", f.read())
    assert m and int(m.group(1)) == IS_BLOCK


def test_engine_requires_the_native_library(monkeypatch, tmp_path):
    # No silent fallback: a missing library is an error that names the build step.
    from bit_consistent_logprob_gb300 import build

    monkeypatch.setattr(_native, "_lib", None)
    monkeypatch.setattr(build, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no CPU or PyTorch fallback"):
        _native.load()


C_CONSUMER = r"""
#include <stdio.h>
#include <string.h>
#include "lp.h"

int main(void) {
    lp_config cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.H = 7168; cfg.V = 129280; cfg.n_leaves = 8; cfg.tp_slices = 1; cfg.max_tokens = 2048;
    unsigned char d[32];
    if (lp_contract_digest(&cfg, LP_PRECISION_BF16, LP_DIGEST_NUMERICAL_POLICY, d) != LP_OK) {
        fprintf(stderr, "%s\n", lp_last_error());
        return 1;
    }
    printf("%d ", lp_version());
    for (int i = 0; i < 32; ++i) printf("%02x", d[i]);
    printf("\n");
    cfg.n_leaves = 3;  /* outside the proven set */
    return lp_contract_digest(&cfg, LP_PRECISION_BF16, 0, d) == LP_ERR_UNSUPPORTED ? 0 : 2;
}
"""


def test_plain_c_program_compiles_and_links_against_the_library(lib, tmp_path):
    # the header is C (not only C++), and a C program links liblp.so with no Python around it
    import shutil
    import subprocess

    from bit_consistent_logprob_gb300 import contract

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("needs gcc")
    src = tmp_path / "consumer.c"
    src.write_text(C_CONSUMER)
    exe = tmp_path / "consumer"
    libdir = os.path.dirname(_native.library_path())
    subprocess.check_call([gcc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                           str(src), "-o", str(exe), "-L", libdir, "-llp",
                           f"-Wl,-rpath,{libdir}"])
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    assert int(out[0]) == lib.lp_version()
    want = contract.digest(contract.NUMERICAL_POLICY, H=7168, V=129280, n_leaves=8,
                           max_tokens=2048)
    assert out[1] == want.hex()
