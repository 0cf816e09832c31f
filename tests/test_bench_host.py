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
        # captured at the full size (scale 1) or on a smaller case scaled by
        # the elements processed
        assert ent["dram_bytes_per_launch"] == ent.get("scale", 16) * ent["captured_bytes"], eng
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


def test_roofline_object_fractions():
    """frac uses the engine's algorithmic bytes; for the fused engine those
    are the DRAM floor 2 p N e (frac == floor_frac); for the executors the
    5 (p - 1) N e element moves, beside which dram_frac (measured bytes) and
    floor_frac are the bounded fractions."""
    p, n, e, peak = 8, 1 << 30, 2, 6657.0
    fused = bench.roofline_object("fused", p, n, e, 5.2, peak, "measured", 33_000_000_000)
    assert fused["frac"] == fused["floor_frac"]
    assert fused["floor_bytes"] == 2 * p * n * e
    assert abs(fused["frac"] - 2 * p * n * e / 5.2e-3 / 1e9 / peak) < 1e-4
    assert abs(fused["dram_frac"] - 33e9 / 5.2e-3 / 1e9 / peak) < 1e-4
    ring = bench.roofline_object("ring", p, n, e, 7.7, peak, "measured", 40_000_000_000)
    assert ring["algorithmic_bytes"] == 5 * (p - 1) * n * e
    assert ring["frac"] > 1.0 > ring["dram_frac"] > ring["floor_frac"]
    assert abs(ring["l2_served"] - (1 - 40e9 / (5 * (p - 1) * n * e))) < 1e-4
    assert "not bounded" in ring["frac_kind"]
    none = bench.roofline_object("tree", p, n, e, 11.0, peak, "fallback", None)
    assert none["dram_frac"] is None and none["l2_served"] is None and none["peak_kind"] == "of fallback"


def test_stored_counters_carry_l2_bytes_and_reach_the_roofline():
    ent = bench.stored_counters("ring", "p8_n1073741824_bf16")
    if ent is None:
        pytest.skip("the ring's code changed since its counters were captured")
    assert ent["dram_bytes_per_launch"] == ent["dram_read_bytes"] + ent["dram_write_bytes"]
    obj = bench.roofline_object("ring", 8, 1 << 30, 2, 7.2, 6657.0, "measured", ent["dram_bytes_per_launch"],
                                ent["lts_bytes_per_launch"])
    assert obj["l2_bytes"] == ent["lts_bytes_per_launch"]
    assert obj["traffic_over_floor"] >= 1.0
