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
    a, b = tmp_path / "k.cu", tmp_path / "h.cu"
    a.write_bytes(b"__global__ void k() {}\n")
    b.write_bytes(b"__global__ void h() {}\n")
    entry = {"sources": {"k.cu": hashlib.sha256(a.read_bytes()).hexdigest(),
                         "h.cu": hashlib.sha256(b.read_bytes()).hexdigest()},
             "bytes": 1234}
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "TRAFFIC", {"kernel": entry})
    w = bench.TRAFFIC_WORKLOAD
    assert bench.traffic_of("kernel", w, None) == 1234
    assert bench.traffic_of("kernel", "other", None) is None       # another workload
    assert bench.traffic_of("kernel", w, "morton") is None         # a variant of the run
    assert bench.traffic_of("unknown", w, None) is None
    b.write_bytes(b"__global__ void h() { }\n")                   # one source changed
    assert bench.traffic_of("kernel", w, None) is None
    b.unlink()
    assert bench.traffic_of("kernel", w, None) is None


def test_traffic_table_names_existing_sources():
    import bench
    for name, t in bench.TRAFFIC.items():
        for src, digest in t["sources"].items():
            assert os.path.exists(os.path.join(ROOT, src)), name
            assert len(digest) == 64, name
        assert t["bytes"] > 0, name


def test_oracle_step_full_and_sampled(capsys):
    """The CPU baseline's oracle step: the whole step, and the sampled step
    that the reference arm and the baseline leg share (a 1/k slice of the
    Gaussians, every k-th non-empty tile in list-length order)."""
    import json
    import types

    import numpy as np

    import bench
    import scenes
    cfg = scenes.make("small_200k_1024x768", n_override=20_000)
    full, wall, stages, text = bench.oracle_step(cfg, 2, 1, {})
    assert full > 0 and wall > 0 and text.startswith("full oracle step")
    assert set(stages) == {"project", "bin", "raster_fwd", "loss", "raster_bwd", "project_bwd",
                           "adam"}
    cache = {}
    s_full, s_wall, _, s_text = bench.oracle_step(cfg, 2, 4, cache)
    assert s_full > s_wall * 0.5 and "every 4th" in s_text
    pr, vals, ranges = cache["full"]
    lens = ranges[:, 1] - ranges[:, 0]
    assert lens.max() > 0 and np.count_nonzero(lens) > 4
    # the reference arm: one JSON line on the host's cores
    args = types.SimpleNamespace(workload="tiny_2k_256", gaussians=None, warmup=1, steps=2)
    bench.reference_arm(args, 0, 1)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["cores"] == bench.host_cores()
    assert line["e2e"]["h2d_bytes_per_step"] == 0
