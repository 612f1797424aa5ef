"""Host logic of the bench's DRAM-traffic record: each kernel's ncu figure
is reported only while the hash of that kernel's own source files matches
the one stored with it, so a change elsewhere in the library leaves it
valid and a change to the kernel voids it."""
import json
import os

import bench


def test_every_timed_kernel_lists_existing_sources():
    csrc = os.path.join(bench.ROOT, "combine_group_limited_gb300", "csrc")
    for kernel, files in bench.KERNEL_SOURCES.items():
        assert files, kernel
        for f in files:
            assert os.path.isfile(os.path.join(csrc, f)), (kernel, f)
        assert len(bench.kernel_source_hash(kernel)) == 16


def test_record_is_used_only_while_its_hash_matches(tmp_path, monkeypatch):
    rec = {"kernels": {
        "combine_kernel": {"source_hash": bench.kernel_source_hash("combine_kernel"), "bytes_per_launch": 123},
        "route_kernel": {"source_hash": "0" * 16, "bytes_per_launch": 456},
    }}
    p = tmp_path / "traffic.json"
    p.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "PROFILE_TRAFFIC", str(p))
    assert bench.recorded_traffic("combine_kernel") == 123
    assert bench.recorded_traffic("route_kernel") is None          # stale hash
    assert bench.recorded_traffic("dispatch_bulk_kernel") is None  # no record
    assert bench.recorded_traffic("not_a_kernel") is None
    p.write_text("not json")
    assert bench.recorded_traffic("combine_kernel") is None


def test_committed_record_names_only_timed_kernels():
    with open(bench.PROFILE_TRAFFIC) as f:
        d = json.load(f)
    for kernel, r in d["kernels"].items():
        assert kernel in bench.KERNEL_SOURCES
        assert r["bytes_per_launch"] > 0 and len(r["source_hash"]) == 16
