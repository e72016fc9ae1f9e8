"""The 3- and 6-bit GEMV code-pair schedules, checked on the host (no GPU).

The fast GEMV path for 3- and 6-bit codes takes its shifts and LOP3 masks from
the tables in ``csrc/qgemv_stream.h``.  ``stream_layout_check.cpp`` compiles
that header with the host compiler, checks every table entry against the
packed layout and replays the path's arithmetic exactly on random chunks
against a bit-by-bit unpack.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "dequant_gemv_gemm_bt_b300", "csrc")


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs a host C++ compiler")
def test_stream_schedules(tmp_path):
    exe = tmp_path / "stream_layout_check"
    subprocess.run(["g++", "-std=c++17", "-O1", "-I", CSRC, os.path.join(HERE, "stream_layout_check.cpp"),
                    "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout
