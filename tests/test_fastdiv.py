"""Host test of the invariant-divisor division used by the GEMV's stream-K partition
(Granlund and Montgomery, "Division by Invariant Integers using Multiplication",
section 4): the header is compiled with the host C++ compiler and compared with plain
unsigned division on about three million (n, d) pairs, edge cases included."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "weight_only_quantised_gb300", "csrc")


def test_fastdiv_matches_division(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = tmp_path / "fastdiv_check"
    subprocess.run([cxx, "-O2", "-std=c++17", "-I", CSRC, "-o", str(exe), os.path.join(HERE, "fastdiv_check.cpp")],
                   check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout + out.stderr
    assert " 0 bad" in out.stdout
