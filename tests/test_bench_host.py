"""Host-side logic of bench.py that needs no GPU: the kernel-source digest
that decides whether a committed DRAM-traffic capture still describes the
kernels, and the traffic lookup built on it."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_code_only_drops_comments_and_spacing():
    src = "int a = 1; // a line comment\n/* a block\n   comment */  float  b;\n"
    assert bench._code_only(src) == "int a = 1; float b;"


def test_code_only_keeps_code_changes():
    assert bench._code_only("x = y + 1;") != bench._code_only("x = y + 2;")
    # a change inside a comment only is not a change
    assert bench._code_only("f(); // old\n") == bench._code_only("f(); // new words\n")



def test_traffic_lookup_follows_the_digest(tmp_path, monkeypatch):
    # a capture is used only while its digest matches the row's sources
    row = "verify"
    good = bench.source_digest(bench.KERNEL_SOURCES[row])
    prof = tmp_path / "profiles"
    prof.mkdir()
    for digest, want in ((good, 123.0), ("0" * 16, None)):
        (prof / "ncu_traffic.json").write_text(json.dumps(
            {row: {"source_digest": digest, "dram_bytes_per_call": 123.0}}))
        monkeypatch.setattr(bench, "ROOT", str(tmp_path))
        monkeypatch.setattr(bench, "source_digest", lambda paths, g=good: g)
        assert bench.traffic_for(row) == want
