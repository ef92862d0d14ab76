"""Host test of the quantiser's division-free quotient (woq_quotient.h, Markstein's correction
step): compiled with the host C++ compiler (no FP contraction) and compared with the
definition, rne of the IEEE fp32 quotient, for every bf16 activation at every bf16 row
maximum from 2^-116 up (all 128 significands of every exponent)."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "weight_only_quantised_gb300", "csrc")


def test_corrected_quotient_gives_the_ieee_code(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = tmp_path / "quotient_check"
    subprocess.run([cxx, "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-I", CSRC, "-o", str(exe),
                    os.path.join(HERE, "quotient_check.cpp")], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=900)
    assert out.returncode == 0, out.stdout + out.stderr
    fields = out.stdout.split()
    checks, t_wrong, bad = int(fields[0]), int(fields[2]), int(fields[7])
    assert bad == 0
    assert checks > 4e8
    assert t_wrong > 1000  # without the correction many codes would differ
