"""bench.py's DRAM-traffic table on CPU: a recorded ncu figure is reported
only while the kernel's sources (comments and blank lines aside) are those
it was captured from, so a changed kernel reports null, not a stale figure."""

import importlib.util
import os

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_traffic_follows_the_kernel_sources(tmp_path, monkeypatch):
    bench = load_bench()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "k.cu").write_text("__global__ void k(int* p) { p[0] = 1; }  // store\n")
    (tmp_path / "k.cuh").write_text("/* helpers */\nconstexpr int kN = 4;\n")
    src = ["k.cu", "k.cuh"]
    traffic = {"w": {"source": src, "sha256": bench.source_sha(src), "bytes_per_launch": 1234},
               "s": {"source": "k.cu", "sha256": bench.source_sha("k.cu"), "scale": 1.5}}
    monkeypatch.setattr(bench, "NCU_TRAFFIC", traffic)
    assert bench.traffic_for("w") == 1234
    assert bench.traffic_for("s", 1000) == 1500.0 and bench.traffic_for("s") is None
    assert bench.traffic_for("missing") is None
    # comments and blank lines do not change the code
    (tmp_path / "k.cu").write_text("// the kernel\n\n__global__ void k(int* p) { p[0] = 1; }\n")
    (tmp_path / "k.cuh").write_text("constexpr int kN = 4;  /* elements */\n\n")
    assert bench.traffic_for("w") == 1234 and bench.traffic_for("s", 1000) == 1500.0
    # a change in a header the kernel includes nulls its figure
    (tmp_path / "k.cuh").write_text("constexpr int kN = 8;\n")
    assert bench.traffic_for("w") is None and bench.traffic_for("s", 1000) == 1500.0
    # so does a change in the kernel, and a missing file
    (tmp_path / "k.cu").write_text("__global__ void k(int* p) { p[0] = 2; }\n")
    assert bench.traffic_for("s", 1000) is None
    os.remove(tmp_path / "k.cu")
    assert bench.traffic_for("s", 1000) is None


def test_recorded_traffic_names_existing_sources():
    # every entry names files that exist, so a figure can only go null by a change
    bench = load_bench()
    for name, rec in bench.NCU_TRAFFIC.items():
        paths = [rec["source"]] if isinstance(rec["source"], str) else rec["source"]
        for p in paths:
            assert os.path.exists(os.path.join(ROOT, p)), (name, p)
        assert ("bytes_per_launch" in rec) != ("scale" in rec), name
