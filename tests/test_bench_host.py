"""Host logic of bench.py that turns device records and committed profile
summaries into the reported figures (no GPU)."""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_only_ignores_comments_and_spacing():
    a = "int x = 1; // first\n/* block\n comment */ int y =  2;\n"
    b = "int x = 1;\nint y = 2; // edited note\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(a.replace("2", "3"))


def test_kernel_source_hash_is_stable_and_distinguishes_kernels():
    h1 = bench.kernel_source_hash("bwd_fused_tc")
    assert h1 == bench.kernel_source_hash("bwd_fused_tc")
    assert len(h1) == 16
    assert h1 != bench.kernel_source_hash("fwd_tc")


def test_tile_pairs_counts_causal_and_full():
    # 3 query tiles x 3 key tiles: 6 pairs on or below the diagonal, 9 in all
    assert bench.tile_pairs(1, 1, 384, causal=True) == 6
    assert bench.tile_pairs(1, 1, 384, causal=False) == 9
    # a ragged tail counts as a tile; batch and heads multiply
    assert bench.tile_pairs(2, 3, 257, causal=True) == 2 * 3 * 6
    # the 128K causal workload: 32 heads x 1024 x 1025 / 2
    assert bench.tile_pairs(1, 32, 131072) == 16_793_600


def test_flops_of_the_workloads():
    fwd, bwd = bench.flops(1, 1, 4, 8, causal=False)
    assert fwd == 4 * 16 * 8 and bwd == 2.5 * fwd
    fwd_c, _ = bench.flops(1, 1, 4, 8, causal=True)
    assert fwd_c == 4 * 10 * 8  # 4 * 5 / 2 visible (query, key) pairs


def test_parse_trace_idle_fraction():
    # one launch, kid 0, 2 CTAs, 5 items: CTA 0 busy [0, 100), CTA 1 [0, 50)
    words = [0, 2, 5, 0, 100, 3, 0, 50, 2]
    (rec,) = bench.parse_trace(words)
    assert rec["kernel"] == "fwd_tc" and rec["ctas"] == 2 and rec["items_run"] == 5
    assert rec["idle_fraction"] == pytest.approx(1 - 150 / 200)
    # two launches back to back, the second perfectly balanced
    (r0, r1) = bench.parse_trace(words + [12, 1, 1, 10, 30, 1])
    assert r1["kernel"] == "bwd_fused_tc" and r1["idle_fraction"] == 0.0
    # a truncated record is dropped, not misread
    assert bench.parse_trace(words[:-1]) == []


def test_recorded_traffic_matches_only_the_current_source(tmp_path, monkeypatch):
    h = bench.kernel_source_hash("bwd_fused_tc")
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "a.md").write_text(
        "text\ntraffic: kernel=bwd_fused_tc source=0000000000000000 d=128 causal=1 bytes=9 units=1\n"
        f"traffic: kernel=bwd_fused_tc source={h} d=64 causal=0 bytes=7 units=1\n"
        f"traffic: kernel=bwd_fused_tc source={h} d=128 causal=1 bytes=1000 units=10\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = bench.recorded_traffic("bwd_fused_tc", 25, 128, True)
    assert rec["bytes"] == pytest.approx(2500.0)  # 100 bytes per unit x 25 units
    assert rec["source"] == os.path.join("profiles", "a.md")
    assert bench.recorded_traffic("bwd_fused_tc", 25, 64, False)["bytes"] == pytest.approx(175.0)
    # another head dimension or masking is another kernel's traffic
    assert bench.recorded_traffic("bwd_fused_tc", 25, 64, True) is None
    assert bench.recorded_traffic("fwd_tc", 25, 128, True) is None


def test_committed_traffic_record_is_well_formed():
    # the committed summary carries one record for the fused backward, whose
    # units are the tile pairs of its capture (64K, 16 heads, causal)
    rec = None
    with open(os.path.join(ROOT, "profiles", "dram_traffic_bwd_fwd_64k.md")) as f:
        for line in f:
            if line.startswith("traffic:"):
                rec = dict(kv.split("=") for kv in line.split()[1:])
    assert rec is not None and rec["kernel"] == "bwd_fused_tc"
    assert rec["d"] == "128" and rec["causal"] == "1"
    assert int(rec["units"]) == bench.tile_pairs(1, 16, 65536)
    assert len(rec["source"]) == 16 and int(rec["bytes"]) > 0
