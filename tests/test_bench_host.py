"""Host logic of bench.py's roofline line (no GPU): the source hash that decides whether the recorded
ncu traffic still belongs to the histogram kernel, and the scaling of a smaller capture's traffic to the
bench's own launches."""
import hashlib
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
bench = pytest.importorskip("bench")


def test_code_only_drops_comments_and_blank_lines_but_keeps_code():
    src = "int a = 1;  // one\n\n/* a block\n   comment */\nint b = a / 2;  /* inline */ int c;\n"
    assert bench._code_only(src) == "int a = 1;\nint b = a / 2;   int c;"
    # a comment edit leaves the hash input unchanged; a code edit does not
    assert bench._code_only(src.replace("// one", "// the first")) == bench._code_only(src)
    assert bench._code_only(src.replace("a / 2", "a / 3")) != bench._code_only(src)


def test_hist_source_hash_is_the_code_of_the_listed_sources():
    h = hashlib.sha256()
    for rel in bench.HIST_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(bench._code_only(f.read()).encode())
    assert bench.hist_source_sha256() == h.hexdigest()


def test_scaled_traffic_follows_the_read_bytes():
    rec = {"dram_bytes_per_launch_captured": 240.0, "read_bytes_per_launch_captured": 200.0}
    assert bench._scaled_traffic(rec, 200.0) == pytest.approx(240.0)
    assert bench._scaled_traffic(rec, 700.0) == pytest.approx(840.0)  # 1.2x the read bytes at any size
    assert bench._scaled_traffic(None, 700.0) is None
    assert bench._scaled_traffic({"dram_bytes_per_launch": 5.0}, 700.0) == 5.0  # an unscaled record


def test_traffic_record_is_used_only_for_its_own_source(tmp_path, monkeypatch):
    rec = {"kernel_source_sha256": bench.hist_source_sha256(), "dram_bytes_per_launch_captured": 1.0,
           "read_bytes_per_launch_captured": 1.0}
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "histogram_traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "hist_source_sha256", lambda: rec["kernel_source_sha256"])
    assert bench._traffic_record() == rec
    monkeypatch.setattr(bench, "hist_source_sha256", lambda: "0" * 64)  # the kernel changed since
    assert bench._traffic_record() is None


def test_code_key_ignores_comments_but_not_code():
    src = "int a = 1;  // one\n/* a\n   block */\n\nint b = a + 2;\n"
    same = "// header\nint a = 1;\n\n\nint b = a + 2;  /* trailing */\n"
    other = "int a = 1;\nint b = a + 3;\n"
    assert bench._code_only(src) == bench._code_only(same)
    assert bench._code_only(src) != bench._code_only(other)
