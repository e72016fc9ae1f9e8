"""Host logic behind bench.py's roofline line (no GPU): the per-launch DRAM
traffic from a committed ncu summary is reported only while the kernel's code
is the code the counters were taken on."""
import os

import bench


def write(path, text):
    os.makedirs(os.path.dirname(path), exist_ok=True)
    with open(path, "w") as f:
        f.write(text)


def test_digest_ignores_comments_and_blank_lines(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    src = os.path.join(tmp_path, "k", "a.cu")
    write(src, "int f(int x) {\n  return x + 1;  // one\n}\n")
    d0 = bench.source_digest(["k/*.cu"])
    write(src, "/* header\n   block */\n\nint f(int x) {\n\n  return x + 1;  // a longer comment\n}\n// end\n")
    assert bench.source_digest(["k/*.cu"]) == d0
    write(src, "int f(int x) {\n  return x + 2;  // one\n}\n")
    assert bench.source_digest(["k/*.cu"]) != d0
    write(os.path.join(tmp_path, "k", "b.cu"), "int g;\n")            # a new file in the set counts
    write(src, "int f(int x) {\n  return x + 1;  // one\n}\n")
    assert bench.source_digest(["k/*.cu"]) != d0


def test_traffic_only_for_the_captured_code(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    write(os.path.join(tmp_path, "profiles", "p.md"),
          "# capture\n\ntraffic_bytes_per_launch: 3.3879e8\nkernel_source_digest: 0123abcd\n")
    assert bench.profile_traffic("p.md", "0123abcd") == 3.3879e8
    assert bench.profile_traffic("p.md", "ffffffff") is None
    assert bench.profile_traffic("missing.md", "0123abcd") is None
    write(os.path.join(tmp_path, "profiles", "q.md"), "traffic_bytes_per_launch: 1e6\n")   # no digest: unusable
    assert bench.profile_traffic("q.md", "0123abcd") is None


def test_peaks_fall_back_only_without_the_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, kind = bench.measured_peaks()
    assert kind == "fallback" and peaks["hbm_gbs"] == 6400.0
    write(os.path.join(tmp_path, "MEASURED_PEAKS.json"), '{"hbm_gbs": 6484.3, "bf16_tflops": 1700.0}')
    peaks, kind = bench.measured_peaks()
    assert kind == "measured" and peaks["hbm_gbs"] == 6484.3
