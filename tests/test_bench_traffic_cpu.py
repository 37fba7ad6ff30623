"""The roofline's `traffic` comes from the committed ncu record (profiles/traffic.json)
only while a kernel's sources are the ones the record was captured on: bench.py hashes
each kernel's source files and reports null once they differ."""

import json
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "online_softmax_07_gb300", "csrc")


def _bench():
    sys.path.insert(0, ROOT)
    import bench
    return bench


def test_kernel_source_lists_name_existing_files():
    bench = _bench()
    for kernel, files in bench.KERNEL_FILES.items():
        assert files, kernel
        for name in files:
            assert os.path.isfile(os.path.join(CSRC, name)), (kernel, name)


def test_traffic_record_entries_are_well_formed():
    bench = _bench()
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    for kernel, ent in rec.items():
        if kernel.startswith("_"):
            continue
        assert kernel in bench.KERNEL_FILES, kernel
        assert isinstance(ent["dram_bytes_per_launch"], int) and ent["dram_bytes_per_launch"] > 0
        assert len(ent["sources"]) == 16
        assert os.path.isfile(os.path.join(ROOT, ent["capture"])), ent["capture"]


def test_changed_sources_give_null_traffic(tmp_path, monkeypatch):
    bench = _bench()
    shutil.copytree(CSRC, tmp_path / "online_softmax_07_gb300" / "csrc")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    record = tmp_path / "profiles" / "traffic.json"
    for kernel, files in bench.KERNEL_FILES.items():
        h = bench.kernel_sources_hash(kernel)
        record.write_text(json.dumps({kernel: {"sources": h, "dram_bytes_per_launch": 123}}))
        assert bench.recorded_traffic(kernel) == 123
        # Any listed file changing (here the last one) makes the record stale.
        src = tmp_path / "online_softmax_07_gb300" / "csrc" / files[-1]
        original = src.read_bytes()
        src.write_bytes(original + b"\n")
        assert bench.kernel_sources_hash(kernel) != h
        assert bench.recorded_traffic(kernel) is None
        src.write_bytes(original)
        assert bench.recorded_traffic(kernel) == 123
    # A missing kernel entry or an unreadable record: null as well.
    record.write_text(json.dumps({}))
    assert bench.recorded_traffic("attn_fwd_tc_kernel") is None
    record.write_text("not json")
    assert bench.recorded_traffic("attn_fwd_tc_kernel") is None
