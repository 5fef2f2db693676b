"""The benchmark's DRAM-traffic record is keyed to the kernel and launch sources (CPU only).

A recorded ncu figure may only be reported while the sources it was measured on are
unchanged; edits to comments or whitespace must not drop it, edits to code must.  Every host
function the key names must exist, or a rename would silently change what is hashed.
"""
import importlib
import json
import os
import re
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture()
def bench(monkeypatch):
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    return importlib.import_module("bench")


def test_every_hashed_host_function_exists(bench):
    with open(os.path.join(ROOT, bench.HOST_LAUNCH[0])) as f:
        src = f.read()
    for name in bench.HOST_LAUNCH[1] + bench.FP8_HOST_LAUNCH:
        text = bench._function_text(src, name)
        assert re.search(r"\b" + re.escape(name) + r"\(", text), name


def test_hash_ignores_comments_and_whitespace_but_not_code(bench, tmp_path, monkeypatch):
    for rel in bench.KERNEL_SOURCES + bench.FP8_SOURCES + [bench.HOST_LAUNCH[0]]:
        os.makedirs(tmp_path / os.path.dirname(rel), exist_ok=True)
        shutil.copy(os.path.join(ROOT, rel), tmp_path / rel)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    base = bench.kernel_source_hash()
    base8 = bench.kernel_source_hash(fp8=True)
    assert re.fullmatch(r"[0-9a-f]{16}", base) and base != base8
    kern = tmp_path / bench.KERNEL_SOURCES[0]
    src = kern.read_text()
    kern.write_text("// a new comment\n/* and a block\n comment */\n" + src.replace("\n", "\n  "))
    assert bench.kernel_source_hash() == base
    kern.write_text(src + "\nconstexpr int kProbeConstant = 1;\n")
    assert bench.kernel_source_hash() != base
    assert bench.kernel_source_hash(fp8=True) != base8


def test_traffic_records_are_well_formed(bench):
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        recs = json.load(f)
    assert {"qwen_prefill", "ds_prefill", "ds_prefill_fp8", "ds_decode_b256"} <= set(recs)
    for key, rec in recs.items():
        assert re.fullmatch(r"[0-9a-f]{16}", rec["kernel_source_sha"]), key
        assert rec["dram_bytes_per_launch"] > 0, key
        assert os.path.exists(os.path.join(ROOT, rec["source"].split(" ")[0])), key


def test_first_rows_keeps_a_prefix_of_the_packed_batch(bench):
    lengths = [300, 500, 200]
    assert bench.first_rows(lengths, 1000) == [300, 500, 200]
    assert bench.first_rows(lengths, 800) == [300, 500]
    assert bench.first_rows(lengths, 650) == [300, 350]
    assert bench.first_rows(lengths, 1) == [1]
    assert sum(bench.first_rows(lengths, 777)) == 777
