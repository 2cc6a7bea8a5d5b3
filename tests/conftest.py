"""Shared pytest configuration.

Markers:
  gpu -- needs a CUDA device (GB300) and the built CUDA library; parity tests
         that compare the CUDA path with the CPU oracle live behind it.
Everything unmarked runs on a CPU-only machine.
"""
import importlib.util
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


# The property-based oracle pins need hypothesis; where it is not installed the
# file is not collected (rather than reported as a skipped module).
collect_ignore = []
if importlib.util.find_spec("hypothesis") is None:
    collect_ignore.append("test_oracle_properties.py")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the built CUDA library")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.lib()
    return oracle
