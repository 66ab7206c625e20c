"""Host logic of the benchmark that needs no GPU: the key under which the
measured DRAM traffic of the fused kernel is stored follows the kernel code and
ignores comment edits, and a record is used only for the code it was taken on."""
from __future__ import annotations

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_code_only_drops_comments_and_spacing():
    a = "int x = 1; // one\n/* a\n block */ float y;\n\n  return x;"
    b = "int x = 1;\nfloat y; return x; // other words"
    assert bench._code_only(a) == bench._code_only(b) == "int x = 1; float y; return x;"


def test_code_only_follows_code():
    assert bench._code_only("a = b + c; // sum") != bench._code_only("a = b - c; // sum")


def test_traffic_is_reported_only_for_the_measured_code(tmp_path, monkeypatch):
    rec = {"source_sha": "0123456789abcdef", "bytes_per_launch_full_workload": 123}
    path = tmp_path / "traffic.json"
    path.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(path))
    assert bench.recorded_traffic("0123456789abcdef") == 123
    assert bench.recorded_traffic("fedcba9876543210") is None
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "missing.json"))
    assert bench.recorded_traffic("0123456789abcdef") is None
