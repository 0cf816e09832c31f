"""Host-side logic of bench.py (no GPU): the roofline bytes per engine, the
comment-insensitive source hash that guards the stored ncu traffic, and the
traffic lookup itself."""
import json
import os

import pytest

import bench
from tests.conftest import ROOT


def test_roofline_bytes_per_engine():
    p, n, e = 8, 1 << 30, 2
    # fused: every rank read once and written once
    assert bench.roofline_bytes("fused", p, n, e) == 2 * p * n * e == 34_359_738_368
    assert bench.roofline_bytes("fused_tree", p, n, e) == 2 * p * n * e
    # schedule executors: 3 moves per reduce-scatter hop, 2 per all-gather hop
    for eng in ("ring", "ring_bidir", "tree"):
        assert bench.roofline_bytes(eng, p, n, e) == 5 * (p - 1) * n * e == 75_161_927_680


def test_code_only_drops_comments_and_blank_lines():
    code = "int a = 1;  // note\n\n/* block\n comment */ int b = 2;\n   \nint c = a + b; /* tail */\n"
    assert bench._code_only(code) == "int a = 1;\n int b = 2;\nint c = a + b;"
    # the same code with other comments hashes the same
    other = "// header\nint a = 1;\n/* x */ int b = 2;\nint c = a + b;\n"
    assert bench._code_only(other).replace(" ", "") == bench._code_only(code).replace(" ", "")


def test_every_engine_source_exists_and_hash_is_stable():
    csrc = os.path.join(ROOT, "ring_all_reduce_rar_gb300", "csrc")
    for eng, files in bench.ENGINE_SOURCES.items():
        for f in files:
            assert os.path.exists(os.path.join(csrc, f)), (eng, f)
        h = bench.kernel_source_hash(eng)
        assert len(h) == 16 and h == bench.kernel_source_hash(eng)


def test_stored_traffic_lookup():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    entries = d["p8_n1073741824_bf16"]
    for eng, ent in entries.items():
        assert ent["dram_bytes_per_launch"] == 16 * ent["captured_bytes"], eng
        got = bench.stored_traffic(eng, "p8_n1073741824_bf16")
        # reported only while the engine's code is the code that was captured
        if ent["kernel_source_hash"] == bench.kernel_source_hash(eng):
            assert got == ent["dram_bytes_per_launch"]
        else:
            assert got is None
    assert bench.stored_traffic("fused", "no_such_workload") is None
    assert bench.stored_traffic("no_such_engine", "p8_n1073741824_bf16") is None


@pytest.mark.parametrize("eng", ["fused", "ring", "tree"])
def test_traffic_below_algorithmic_bytes(eng):
    """DRAM traffic above the algorithmic bytes would mean re-reads; every
    stored capture is at or below them (L2 serves the rest)."""
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        ent = json.load(f)["p8_n1073741824_bf16"][eng]
    assert 0 < ent["dram_bytes_per_launch"] <= bench.roofline_bytes(eng, 8, 1 << 30, 2)
