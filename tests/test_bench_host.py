"""Host logic of bench.py that needs no GPU: the DRAM-traffic records that the
roofline object quotes are matched by kernel and workload, and dropped once
the kernel's source has changed since the capture."""
import hashlib
import json
import os

import bench


def _tree(tmp_path, records, src_text=b"// kernel source\n"):
    csrc = tmp_path / "long_context_masked_mask_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_bytes(src_text)
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "traffic.json").write_text(json.dumps(records))
    return hashlib.sha256(src_text).hexdigest()


def _rec(sha, workload, nbytes):
    return {"source": "k.cu", "source_sha256": sha, "workload": workload, "launch": f"{workload} launch",
            "dram_bytes_per_launch": nbytes}


def test_traffic_record_per_workload(tmp_path, monkeypatch):
    sha = hashlib.sha256(b"// kernel source\n").hexdigest()
    _tree(tmp_path, {"k_kernel": [_rec(sha, "w1", 10), _rec(sha, "w2", 20)]})
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_lookup("k_kernel", "w1")["bytes"] == 10
    assert bench.traffic_lookup("k_kernel", "w2")["bytes"] == 20
    assert bench.traffic_lookup("k_kernel", "w3") is None
    assert bench.traffic_lookup("other_kernel", "w1") is None


def test_traffic_single_record_form(tmp_path, monkeypatch):
    sha = hashlib.sha256(b"// kernel source\n").hexdigest()
    _tree(tmp_path, {"k_kernel": _rec(sha, "w1", 7)})
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_lookup("k_kernel", "w1")["bytes"] == 7


def test_traffic_dropped_when_source_changed(tmp_path, monkeypatch):
    _tree(tmp_path, {"k_kernel": [_rec("0" * 64, "w1", 10)]})
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_lookup("k_kernel", "w1") is None


def test_committed_traffic_records_are_well_formed():
    path = os.path.join(bench.ROOT, "profiles", "traffic.json")
    data = json.load(open(path))
    for kernel, recs in data.items():
        for r in recs if isinstance(recs, list) else [recs]:
            assert os.path.exists(os.path.join(bench.ROOT, "long_context_masked_mask_gb300", "csrc",
                                               r["source"])), kernel
            assert len(r["source_sha256"]) == 64 and r["workload"] and r["launch"]
            assert r["dram_bytes_per_launch"] > 0
