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
    write(os.path.join(tmp_path, "profiles", "p.json"),
          '{"traffic_bytes_per_launch": 3.3879e8, "kernel_source_digest": "0123abcd"}')
    assert bench.profile_traffic("p.json", "0123abcd") == 3.3879e8
    assert bench.profile_traffic("p.json", "ffffffff") is None
    assert bench.profile_traffic("missing.json", "0123abcd") is None
    write(os.path.join(tmp_path, "profiles", "q.json"), '{"traffic_bytes_per_launch": 1e6}')   # no digest
    assert bench.profile_traffic("q.json", "0123abcd") is None
    write(os.path.join(tmp_path, "profiles", "r.json"), "not json")
    assert bench.profile_traffic("r.json", "0123abcd") is None


def test_oracle_baseline_runs_on_spawned_workers():
    """The CPU baseline spreads the pass's projections over spawned workers (one
    per core asked for) and counts the bytes every worker processed."""
    shapes = [("a", 64, 128), ("b", 32, 256), ("c", 16, 64)]
    rate, nbytes, count, procs = bench.oracle_rate("bench-host-test", shapes, 0.3, procs=2)
    assert procs == 2 and count >= 2 and nbytes > 0 and rate > 0
    assert bench.oracle_rate("bench-host-test", shapes[:1], 0.1, procs=4)[3] == 1   # never more workers than projections
    ncpu, naff = bench.host_cores()
    assert 1 <= naff <= ncpu


def test_peaks_fall_back_only_without_the_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, kind = bench.measured_peaks()
    assert kind == "fallback" and peaks["hbm_gbs"] == 6400.0
    write(os.path.join(tmp_path, "MEASURED_PEAKS.json"), '{"hbm_gbs": 6484.3, "bf16_tflops": 1700.0}')
    peaks, kind = bench.measured_peaks()
    assert kind == "measured" and peaks["hbm_gbs"] == 6484.3
