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


# ---- the roofline's algorithmic work, against closed forms --------------
# Per visible (query row, key): 2*576 flop for the score and 2*512 for the
# output (2176).  Bytes: every cache row once (1152 B bf16, 576 B e4m3, the
# shared prefix pages once), the queries (576 bf16 values per row), out (512
# bf16), lse (fp32), the page-table entries read and the lengths.

def _shape_only(seq_lens, H, Q, page_table, kv_dtype="bf16"):
    from types import SimpleNamespace

    import numpy as np

    return SimpleNamespace(batch=len(seq_lens), num_heads=H, q_len=Q, kv_dtype=kv_dtype,
                           seq_lens=np.asarray(seq_lens, dtype=np.int32), page_table=np.asarray(page_table))


def test_algorithmic_work_kimi_closed_form():
    import numpy as np

    B, H, L = 64, 64, 8192
    table = np.random.default_rng(0).permutation(B * 128).reshape(B, 128)
    nbytes, flops, rows = bench.algorithmic_work(_shape_only([L] * B, H, 1, table))
    assert rows == B * L
    assert flops == B * L * H * 2176  # 73.1 GFLOP
    assert nbytes == B * L * 1152 + B * H * (1152 + 1024 + 4) + B * 128 * 4 + B * 4  # 612.9 MB


def test_algorithmic_work_causal_drafts_and_e4m3():
    import numpy as np

    lens, H, Q = [10, 100], 16, 2
    table = np.array([[5, -1], [0, 1]])
    nbytes, flops, rows = bench.algorithmic_work(_shape_only(lens, H, Q, table, "fp8_e4m3"))
    # draft i sees L - Q + i + 1 keys: 2L - 1 per request over the two drafts
    assert flops == ((2 * 10 - 1) + (2 * 100 - 1)) * H * 2176
    assert rows == 110
    assert nbytes == 110 * 576 + 2 * Q * H * (1152 + 1024 + 4) + 3 * 4 + 2 * 4


def test_algorithmic_work_counts_shared_prefix_pages_once():
    import numpy as np

    # three requests share pages 7, 8 (128 tokens), then private suffixes
    lens = [128 + 10, 128 + 64, 128 + 65]
    table = np.array([[7, 8, 0, -1], [7, 8, 1, -1], [7, 8, 2, 3]])
    nbytes, flops, rows = bench.algorithmic_work(_shape_only(lens, 16, 1, table))
    assert rows == 128 + 10 + 64 + 65
    assert flops == sum(lens) * 16 * 2176
    assert nbytes == rows * 1152 + 3 * 16 * (1152 + 1024 + 4) + (3 + 3 + 4) * 4 + 3 * 4


def test_reference_arm_prints_the_contract_line():
    import subprocess

    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["steps"] == 1 and line["warmup"] == 3
    assert line["config"]["workload"] == "tiny" and line["value"] > 0
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1 and cb["sample"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
