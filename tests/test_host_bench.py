"""Host logic of the benchmark that needs no GPU: the roofline's `traffic` comes from a
committed ncu capture only while that capture's source hash matches the current kernel and
planner sources."""

import json
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _tree(tmp_path):
    """A copy of the kernel sources under a scratch root, with an empty profiles folder."""
    csrc = tmp_path / "prefix_shared_kv_token_gb300" / "csrc"
    shutil.copytree(os.path.join(ROOT, "prefix_shared_kv_token_gb300", "csrc"), csrc)
    (tmp_path / "profiles").mkdir()
    return tmp_path, csrc


def test_traffic_follows_the_source_hash(tmp_path, monkeypatch):
    root, csrc = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    h = bench.kernel_hash("decode")
    path = root / "profiles" / "decode_some_workload.json"
    path.write_text(json.dumps({"source_hash": h, "dram_bytes_per_launch": 123456789.0}))
    assert bench.profiled_traffic("decode", "some_workload") == 123456789.0
    # no capture for another workload or kind
    assert bench.profiled_traffic("decode", "other_workload") is None
    assert bench.profiled_traffic("extend", "some_workload") is None
    # any change to a source the decode call runs (or plans with) makes the capture stale
    for name in ("attn_decode.cu", "attn_extend.cu", "plan.cpp", "common.cuh"):
        f = csrc / name
        old = f.read_text()
        f.write_text(old + "\n// changed\n")
        assert bench.profiled_traffic("decode", "some_workload") is None, name
        f.write_text(old)
    assert bench.profiled_traffic("decode", "some_workload") == 123456789.0
    # a source outside the decode call does not
    f = csrc / "kv_store.cu"
    f.write_text(f.read_text() + "\n// changed\n")
    assert bench.profiled_traffic("decode", "some_workload") == 123456789.0


def test_extend_hash_ignores_the_decode_kernel(tmp_path, monkeypatch):
    root, csrc = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    h = bench.kernel_hash("extend")
    f = csrc / "attn_decode.cu"
    f.write_text(f.read_text() + "\n// changed\n")
    assert bench.kernel_hash("extend") == h
    f = csrc / "attn_extend.cu"
    f.write_text(f.read_text() + "\n// changed\n")
    assert bench.kernel_hash("extend") != h


def test_committed_captures_name_their_workload_and_command():
    prof = os.path.join(ROOT, "profiles")
    found = [n for n in os.listdir(prof) if n.endswith(".json")]
    assert found
    for name in found:
        with open(os.path.join(prof, name)) as fh:
            d = json.load(fh)
        kind, workload = name[:-5].split("_", 1)
        assert kind in ("extend", "decode") and d["workload"] == workload
        assert d["dram_bytes_per_launch"] > 0 and len(d["source_hash"]) == 16
        assert "--clock-control none" in d["command"] and "bench.py" in d["command"]
