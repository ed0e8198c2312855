"""Shared pytest configuration.

``-m gpu`` tests need a CUDA device and the built library; everything else runs
on the CPU (oracle pins, host logic, library symbol checks).
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the built CUDA library")


def read_golden(name: str) -> dict:
    """Parse a tests/golden/*.txt fixture: 'key = value' lines, '#' comments."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            parts = v.split()
            vals = [float(p) for p in parts]
            out[k] = vals[0] if len(vals) == 1 else vals
    return out


@pytest.fixture(scope="session")
def golden():
    return read_golden
