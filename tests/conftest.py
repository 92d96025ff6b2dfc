"""Shared test configuration.

Markers:
  gpu  -- needs a CUDA device and the compiled GPU library (run with -m gpu).
Everything unmarked runs on a CPU-only machine.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the compiled library")


def read_golden(name):
    """Parse a tests/golden/*.txt fixture: ``key: v1 v2 ...`` lines, '#' comments.

    Returns {key: (values as floats, decimals printed per value)}.
    """
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, vals = line.split(":", 1)
            toks = vals.split()
            decs = [len(t.split(".", 1)[1]) if "." in t and "e" not in t.lower() else 0
                    for t in toks]
            out[key.strip()] = ([float(t) for t in toks], decs)
    return out


@pytest.fixture
def golden_file():
    return read_golden
