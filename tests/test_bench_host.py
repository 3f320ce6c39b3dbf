"""bench.py's host-side accounting on CPU: the algorithmic bytes a decode
reads per format and workload, the rows a windowed T-row decode sees, and
the source hash that decides whether recorded ncu traffic still applies."""

import json
import os
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from quantized_kv_cache_08_gb300.inputs import workload  # noqa: E402


def test_bytes_per_row_by_format():
    wl = workload("ctx32k")                       # 8 KV heads x 128 = 32 blocks per row
    assert bench.kv_bytes_per_row(wl) == 32 * (34 + 24) == 1856
    assert bench.kv_bytes_per_row(wl, "e4m3") == 32 * 64 == 2048
    assert bench.kv_bytes_per_row(workload("swa_ring")) == 16 * 58   # 8 x 64


def test_algorithmic_bytes_of_the_workloads():
    wl = workload("ctx32k")
    lens = bench.decode_lengths(wl)
    assert sum(bench.visible_rows(wl, L) for L in lens) * bench.kv_bytes_per_row(wl) == 60_817_408
    ring = workload("swa_ring")
    lens = bench.decode_lengths(ring)
    assert lens == [2 * ring.window]
    # a T=1 row sees its own row and the window - 1 before it
    assert bench.visible_rows(ring, lens[0]) == ring.window
    assert bench.visible_rows(ring, lens[0]) * bench.kv_bytes_per_row(ring) == 3_801_088
    spec = workload("spec_verify")                # T = 8, no window: every row
    assert bench.visible_rows(spec, 16384) == 16384


def test_visible_rows_union_of_causal_windows():
    wl = workload("spec_verify", window=100)      # T = 8 query rows
    # row t sees [L-T+t+1-100, L-T+t+1); the union starts at the first row's start
    assert bench.visible_rows(wl, 1000) == 100 + 8 - 1
    assert bench.visible_rows(wl, 50) == 50


def _copy_tree(tmp_path):
    root = tmp_path / "r"
    shutil.copytree(os.path.join(ROOT, "quantized_kv_cache_08_gb300", "csrc"),
                    root / "quantized_kv_cache_08_gb300" / "csrc")
    (root / "profiles").mkdir()
    return root


def test_source_hash_ignores_comments_only(tmp_path, monkeypatch):
    root = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    h0 = bench.kernel_source_hash()
    f = root / "quantized_kv_cache_08_gb300" / "csrc" / "kvq_append.cu"
    src = f.read_text()
    f.write_text("// a new comment line\n" + src.replace("namespace kvq {", "namespace kvq {  /* note */", 1))
    assert bench.kernel_source_hash() == h0
    f.write_text(src.replace("atomicExch(err_d, kErrCounter);", "atomicExch(err_d, kErrWait);", 1))
    assert bench.kernel_source_hash() != h0


def test_recorded_traffic_only_for_matching_sources(tmp_path, monkeypatch):
    root = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(root))
    h = bench.kernel_source_hash()
    rec = {"ctx32k": {"source_hash": h, "dram_bytes_per_decode": 123},
           "ctx32k:e4m3": {"source_hash": "0" * 16, "dram_bytes_per_decode": 456}}
    (root / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic("ctx32k") == 123
    assert bench.recorded_traffic("ctx32k:e4m3") is None
    assert bench.recorded_traffic("batch64") is None


def test_committed_traffic_matches_current_sources():
    """profiles/traffic.json was captured on the kernel code as it stands."""
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
        rec = json.load(fh)
    for name in ("ctx32k", "ctx32k:e4m3"):
        assert rec[name]["source_hash"] == bench.kernel_source_hash(), name
        assert bench.recorded_traffic(name) == rec[name]["dram_bytes_per_decode"]
        # DRAM reads of the split kernel within 1% of the algorithmic bytes
        alg = rec[name]["algorithmic_bytes_per_decode"]
        assert alg <= rec[name]["split_kernel"]["dram_bytes_read"] <= 1.01 * alg


@pytest.mark.parametrize("fmt", sorted(bench.FORMATS))
def test_formats_known_to_the_cache(fmt):
    from quantized_kv_cache_08_gb300.cache import KVCache
    assert fmt in KVCache.FORMATS
    assert KVCache.FORMATS[fmt][2] + KVCache.FORMATS[fmt][3] == bench.FORMATS[fmt][1]


def test_traffic_key_separates_kernel_and_shape_options():
    import argparse
    a = argparse.Namespace(softcap=0.0, t=0)
    assert bench.traffic_key("ctx32k", "q8_0/q5_1", a) == "ctx32k"
    assert bench.traffic_key("ctx32k", "e4m3", a) == "ctx32k:e4m3"
    assert bench.traffic_key("ctx32k", "q8_0/q5_1", argparse.Namespace(softcap=3.0, t=0)) == "ctx32k:softcap"
    assert bench.traffic_key("swa_ring", "q8_0/q5_1", argparse.Namespace(softcap=0.0, t=8)) == "swa_ring:T8"


def test_reference_arm_with_query_rows_and_softcap(capsys):
    """--impl reference runs the oracle on CPU; --t and --softcap reach it."""
    import argparse
    args = argparse.Namespace(workload="ctx512", t=4, softcap=2.0, kv_format="q8_0/q5_1", steps=1,
                              warmup=200)
    line = bench.run_reference(args, 1, 0)
    assert line["config"]["T"] == 4 and line["config"]["softcap"] == 2.0
    assert line["value"] > 0 and "512 visible rows" in line["cpu_baseline"]["sample"]
