"""Host-side accounting of bench.py, on the CPU: the DRAM traffic figure is
reported only for the exact kernel source it was captured on, and only for
its workload and the default variant."""
import hashlib
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def test_traffic_only_for_the_captured_source(tmp_path, monkeypatch):
    import bench
    src = tmp_path / "k.cu"
    src.write_bytes(b"__global__ void k() {}\n")
    entry = {"source": "k.cu", "sha256": hashlib.sha256(src.read_bytes()).hexdigest(),
             "workload": "ring", "bytes": 1234}
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "TRAFFIC", {"kernel": entry})
    assert bench.traffic_of("kernel", "ring", None) == 1234
    assert bench.traffic_of("kernel", "other", None) is None       # another workload
    assert bench.traffic_of("kernel", "ring", "morton") is None     # a variant of the run
    assert bench.traffic_of("unknown", "ring", None) is None
    src.write_bytes(b"__global__ void k() { }\n")                   # the source changed
    assert bench.traffic_of("kernel", "ring", None) is None
    src.unlink()
    assert bench.traffic_of("kernel", "ring", None) is None


def test_traffic_table_names_existing_sources():
    import bench
    for name, t in bench.TRAFFIC.items():
        assert os.path.exists(os.path.join(ROOT, t["source"])), name
        assert len(t["sha256"]) == 64 and t["bytes"] > 0, name
