import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workloads")


def pytest_sessionstart(session):
    # Build the CUDA library (nvcc, sm_103a) and the C oracle (gcc) when their
    # sources are newer than the built files, so that every test module imports
    # the library as built from this tree.
    from block_scaled_fp4_persistent_gb300 import _build
    _build.build()
    import oracle
    oracle.build()
