"""Host-side pieces of the benchmark: the profiled-traffic record is used only
while the kernel sources are the ones that were profiled."""
import json
import os
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _copy_tree(dst):
    rec = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    for f in rec["sources"] + ["profiles/traffic.json"]:
        os.makedirs(os.path.join(dst, os.path.dirname(f)), exist_ok=True)
        shutil.copy(os.path.join(ROOT, f), os.path.join(dst, f))
    return rec


def test_traffic_record_follows_the_sources(tmp_path, monkeypatch):
    if not os.path.exists(os.path.join(ROOT, "profiles", "traffic.json")):
        pytest.skip("no traffic record")
    rec = _copy_tree(str(tmp_path))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    expected = bench.profiled_traffic("kimi")
    assert expected in (None, rec["dram_bytes_per_launch"]["kimi"])
    assert bench.profiled_traffic("no-such-batch") is None
    # any edit of a profiled source voids the record
    src = os.path.join(str(tmp_path), rec["sources"][0])
    with open(src, "a") as f:
        f.write("\n// edited\n")
    assert bench.profiled_traffic("kimi") is None


def test_missing_record_gives_none(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("kimi") is None
