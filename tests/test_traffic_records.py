"""The ncu traffic records under profiles/ are reported by the bench only while the
kernel source they were taken from is unchanged (CPU only)."""
from __future__ import annotations

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _tree(tmp_path, kernel_body: str, comment: str = "") -> None:
    csrc = tmp_path / "memory_bound_decode_dequant_gb300" / "csrc"
    csrc.mkdir(parents=True, exist_ok=True)
    (tmp_path / "include").mkdir(exist_ok=True)
    (tmp_path / "profiles").mkdir(exist_ok=True)
    (tmp_path / "include" / "api.h").write_text("int api(void);\n")
    (csrc / "util.cuh").write_text('#include "../../include/api.h"\n// helper\ninline int two() { return 2; }\n')
    (csrc / "k.cu").write_text(f'#include "util.cuh"\n/* {comment} */\n{kernel_body}\n')


def _use(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "CSRC", str(tmp_path / "memory_bound_decode_dequant_gb300" / "csrc"))


def test_digest_follows_code_not_comments(monkeypatch, tmp_path):
    _use(monkeypatch, tmp_path)
    _tree(tmp_path, "int k() { return two(); }", "first")
    d0 = bench.source_digest("k.cu")
    _tree(tmp_path, "int k()  {\n  return two();\n}", "a reworded comment")
    assert bench.source_digest("k.cu") == d0
    _tree(tmp_path, "int k() { return two() + 1; }")
    assert bench.source_digest("k.cu") != d0
    # a change in an included header changes it too
    _tree(tmp_path, "int k() { return two(); }")
    (tmp_path / "include" / "api.h").write_text("int api(int);\n")
    assert bench.source_digest("k.cu") != d0


def test_stale_or_unlabelled_record_reads_as_null(monkeypatch, tmp_path):
    _use(monkeypatch, tmp_path)
    _tree(tmp_path, "int k() { return two(); }")
    rec = {"bytes_per_launch": 1234, "translation_unit": "k.cu", "source_digest": bench.source_digest("k.cu")}
    path = tmp_path / "profiles" / "k.traffic.json"
    path.write_text(json.dumps(rec))
    assert bench.read_traffic("k") == 1234
    _tree(tmp_path, "int k() { return 3; }")
    assert bench.read_traffic("k") is None
    path.write_text(json.dumps({"bytes_per_launch": 1234}))
    assert bench.read_traffic("k") is None
    assert bench.read_traffic("missing") is None


def test_committed_records_name_their_source():
    prof = os.path.join(ROOT, "profiles")
    recs = [f for f in os.listdir(prof) if f.endswith(".traffic.json")]
    assert recs
    for f in recs:
        with open(os.path.join(prof, f)) as fh:
            rec = json.load(fh)
        assert rec["bytes_per_launch"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
        assert os.path.exists(os.path.join(bench.CSRC, rec["translation_unit"]))
        assert len(rec["source_digest"]) == 16
