import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


def pytest_sessionstart(session):
    # Build the CUDA library (nvcc cross-compiles without a GPU) and the oracle when stale.
    # The build script runs as a program so that a missing library does not break the import.
    subprocess.run([sys.executable, os.path.join(ROOT, "weight_only_quantised_gb300", "_build.py")], check=True,
                   stdout=subprocess.DEVNULL)
    import oracle
    oracle.build()
