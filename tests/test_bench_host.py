"""Host logic of the benchmark that needs no GPU: the committed DRAM-traffic
records are reported only while the kernel sources they were taken on are
unchanged, and only for their own kernel and workload."""
import json

import bench


def _tree(tmp_path, text):
    csrc = tmp_path / "paged_hybrid_sliding_gb300" / "csrc"
    csrc.mkdir(parents=True, exist_ok=True)
    (csrc / "k.cu").write_text(text)
    (tmp_path / "profiles").mkdir(exist_ok=True)


def test_traffic_record_follows_source_hash(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _tree(tmp_path, "kernel v1")
    h = bench.kernel_source_hash(("k.cu",))
    rec = {"entries": [{"kernel": "phs_k", "workload": "w64", "sources": ["k.cu"],
                        "source_hash": h, "dram_bytes_per_launch": 4096}]}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic("phs_k", "w64") == 4096
    assert bench.recorded_traffic("phs_k", "w16") is None       # another workload
    assert bench.recorded_traffic("phs_other", "w64") is None   # another kernel
    _tree(tmp_path, "kernel v2")                                # the source changed
    assert bench.kernel_source_hash(("k.cu",)) != h
    assert bench.recorded_traffic("phs_k", "w64") is None


def test_traffic_record_missing_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.recorded_traffic("phs_k", "w64") is None


def test_committed_records_name_existing_sources():
    # every committed record hashes files that exist in the kernel sources
    with open(f"{bench.ROOT}/profiles/traffic.json") as f:
        rec = json.load(f)
    assert rec["entries"]
    for e in rec["entries"]:
        bench.kernel_source_hash(e["sources"])  # raises if a file is missing
        assert e["dram_bytes_per_launch"] > 0
